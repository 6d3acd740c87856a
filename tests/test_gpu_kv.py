"""GPU parity of kv_rmsnorm_rope_cache against the float64 oracle on the same
seeded inputs: every cache byte outside the indexed rows bit-exact, 16-bit
outputs within 2**-7*|ref| + 1e-6, 8-bit codes within one code, and every
code bit-identical to the oracle's wherever its float64 value lies farther
than 2**-17 (relative) from a rounding boundary; device status bits equal. Covers the four KV workloads at full size, both kernel
paths (vectorised and generic), every cache mode and code type, strided and
misaligned rows, and the degenerate cases."""
import numpy as np
import pytest
import torch

from attention_prologue_kv_gb300 import workloads as wl
from helpers import (check_robust_kv, codes_of, compare_cache, guarded_cache, run_gpu_kv, run_oracle_kv,
                     sentinel_cache)

pytestmark = pytest.mark.gpu


def check(case, **kw):
    ref_ckv, ref_k, ref_st = run_oracle_kv(case)
    g_ckv, g_k, g_st = run_gpu_kv(case, **kw)
    assert g_st == ref_st
    n1, ex1 = compare_cache(g_ckv, ref_ckv, case.ckv_dtype, case.Dv)
    n2, ex2 = compare_cache(g_k, ref_k, case.k_dtype, case.Dk)
    assert n1 == n2
    if n1:
        check_robust_kv(case, g_ckv, g_k)
    return n1, ex1, ex2


@pytest.mark.parametrize("make", [wl.tiny_norm, wl.decode_paged, wl.prefill_paged, wl.quant_fp8],
                         ids=["tiny_norm", "decode_paged", "prefill_paged", "quant_fp8"])
def test_workloads_full_size(make):
    case = make()
    n, ex_ckv, ex_k = check(case)
    assert n == case.active_tokens()
    # one rounding on each side: nearly every element is bit-identical
    assert ex_ckv > 0.97 and ex_k > 0.97


@pytest.mark.parametrize("Dv,Dk", [(512, 64), (24, 16), (256, 8), (1024, 256), (520, 72),
                                   (6, 2), (1032, 64), (512, 258), (10, 6), (1, 2)])
def test_shapes_vector_and_generic_paths(Dv, Dk):
    case = wl.make_kv_case("s", 3, 37, Dv=Dv, Dk=Dk, mode="PA_BSND", d0=40, d1=4, seed=Dv * 7 + Dk,
                           skip=5)
    check(case)


@pytest.mark.parametrize("mode", ["Norm", "PA_BSND", "PA_BLK_BSND"])
@pytest.mark.parametrize("d1", [1, 3, 128])
def test_cache_modes_ragged(mode, d1):
    T_B, T_S = 5, 203
    d0 = {"Norm": 7, "PA_BSND": -(-T_B * T_S // d1) + 3, "PA_BLK_BSND": T_B * -(-T_S // d1) + 2}[mode]
    if mode == "Norm":
        d1 = max(d1, T_S) + 1
    case = wl.make_kv_case("m", T_B, T_S, mode=mode, d0=d0, d1=d1, seed=31 + d1, skip=3)
    check(case)


@pytest.mark.parametrize("ckv,k", [("int8", "bf16"), ("fp8_e4m3fn", "bf16"), ("fp8_e5m2", "bf16"),
                                   ("bf16", "int8"), ("bf16", "fp8_e4m3fn"), ("bf16", "fp8_e5m2"),
                                   ("int8", "int8"), ("fp8_e4m3fn", "fp8_e4m3fn"),
                                   ("fp8_e5m2", "fp8_e4m3fn")])
@pytest.mark.parametrize("per_tensor", [False, True])
def test_quantisation_scenarios(ckv, k, per_tensor):
    kw = dict(scale_len=1, k_scale_len=1) if per_tensor else {}
    case = wl.make_kv_case("q", 16, 33, mode="PA_BSND", d0=8, d1=128, ckv_dtype=ckv, k_dtype=k,
                           seed=41, skip=4, kv_std=3.0, **kw)
    check(case)


def test_quantisation_generic_path():
    case = wl.make_kv_case("q", 4, 9, Dv=20, Dk=6, mode="PA_BSND", d0=4, d1=16,
                           ckv_dtype="fp8_e4m3fn", k_dtype="int8", seed=42)
    check(case)


def test_fp16_inputs_and_caches():
    case = wl.make_kv_case("h", 6, 50, mode="Norm", d0=8, d1=64, ckv_dtype="f16", k_dtype="f16",
                           in_dtype="f16", seed=43, skip=7)
    check(case)
    case = wl.make_kv_case("h", 6, 50, mode="PA_BSND", d0=8, d1=64, ckv_dtype="fp8_e4m3fn",
                           k_dtype="f16", in_dtype="f16", seed=44)
    check(case)


def test_kc_scale():
    case = wl.make_kv_case("a", 4, 64, mode="PA_BSND", d0=4, d1=64, seed=45, kc_scale=0.3)
    check(case)
    case = wl.make_kv_case("a", 4, 64, mode="PA_BSND", d0=4, d1=64, seed=46, kc_scale=2.5,
                           ckv_dtype="fp8_e4m3fn")
    check(case)


@pytest.mark.parametrize("pad", [64, 3])
def test_strided_rows(pad):
    """kv as a column slice of wider rows (vectorised when the stride keeps 16-byte rows)."""
    case = wl.make_kv_case("w", 7, 40, mode="PA_BSND", d0=4, d1=128, seed=47, row_pad=pad)
    assert not case.kv.is_contiguous()
    check(case)


def test_index_length_is_checked_against_the_cache_mode():
    """The kernels read one index entry per token (one per BlockSize tokens in
    PA_BLK_BSND); a shorter index is refused before launch."""
    import attention_prologue_kv_gb300 as kvr
    case = wl.make_kv_case("x", 3, 20, mode="PA_BLK_BSND", d0=12, d1=8, seed=67)
    assert case.index.numel() == 3 * 3
    ckv = sentinel_cache(case.cache_shapes()[0], "bf16")
    k = sentinel_cache(case.cache_shapes()[1], "bf16")
    args = (case.kv.cuda(), case.gamma.cuda(), case.cos.cuda(), case.sin.cuda())
    with pytest.raises(ValueError):
        kvr.kv_rmsnorm_rope_cache(*args, case.index[:8].cuda(), ckv, k, cache_mode="PA_BLK_BSND")
    with pytest.raises(ValueError):   # cos shorter than one entry row per token
        kvr.kv_rmsnorm_rope_cache(args[0], args[1], args[2][:2].contiguous(), args[3], case.index.cuda(), ckv, k,
                                  cache_mode="PA_BLK_BSND")
    with pytest.raises(ValueError):   # the flattened (T, D) form implies one entry per token
        kvr.kv_rmsnorm_rope_cache(args[0].view(60, -1), args[1], args[2].view(60, -1), args[3].view(60, -1),
                                  case.index.cuda(), ckv, k, cache_mode="PA_BLK_BSND")


@pytest.mark.parametrize("mode,pad", [("PA_BSND", 0), ("PA_BSND", 64), ("Norm", 0), ("Norm", 3)])
def test_token_flattened_2d_form(mode, pad):
    """The token-flattened shapes of the MLA page's BS fusion: kv (T, D) (dense,
    or a column slice of wider rows), cos/sin (T, Dk), index (T). Each token
    is one row: in PA_BSND it goes to slot index[t] (the same as in the 4-D
    form); in Norm mode token t is batch t of the cache, row index[t]. Full
    decode size in PA_BSND (256 tokens, 4096 x 128 slots), compared element
    by element with the oracle."""
    import attention_prologue_kv_gb300 as kvr
    if mode == "PA_BSND":
        case = wl.make_kv_case("t2", 256, 1, mode="PA_BSND", d0=4096, d1=128, seed=1302, skip=5,
                               row_pad=pad)
    else:
        case = wl.make_kv_case("t2", 96, 1, mode="Norm", d0=100, d1=16, seed=1303, skip=7, row_pad=pad)
    T, D, Dk = case.T, case.Dv + case.Dk, case.Dk
    kv2 = case.meta["wide"].cuda()[:, :D]
    assert kv2.dim() == 2 and kv2.shape == (T, D) and kv2.is_contiguous() == (pad == 0)
    ckv, c1 = guarded_cache(case.cache_shapes()[0], "bf16")
    k, c2 = guarded_cache(case.cache_shapes()[1], "bf16")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvr.kv_rmsnorm_rope_cache(kv2, case.gamma.cuda(), case.cos.reshape(T, Dk).cuda(),
                              case.sin.reshape(T, Dk).cuda(), case.index.reshape(T).cuda(), ckv, k,
                              cache_mode=mode, eps=case.eps, dev_status=status)
    torch.cuda.synchronize()
    c1()
    c2()
    ref_ckv, ref_k, ref_st = run_oracle_kv(case)
    assert int(status.item()) == ref_st == 0
    n1, _ = compare_cache(codes_of(ckv), ref_ckv, "bf16", case.Dv)
    n2, _ = compare_cache(codes_of(k), ref_k, "bf16", case.Dk)
    assert n1 == n2 == case.active_tokens()


def test_misaligned_pointers_take_the_generic_path():
    case = wl.make_kv_case("u", 5, 11, mode="PA_BSND", d0=2, d1=64, seed=48)
    T, D = case.T, case.Dv + case.Dk
    buf = torch.empty(T * D + 1, dtype=torch.bfloat16, device="cuda")
    kv = buf[1:].view(case.Bkv, 1, case.Skv, D)
    kv.copy_(case.kv.cuda())
    assert kv.data_ptr() % 16 != 0
    check(case, kv=kv)


def test_out_of_range_indices_are_skipped_and_flagged():
    case = wl.make_kv_case("r", 4, 32, mode="PA_BSND", d0=8, d1=16, seed=49)
    case.index[3] = 8 * 16
    case.index[17] = -5
    case.index[30] = 1 << 40
    ref_ckv, ref_k, ref_st = run_oracle_kv(case)
    assert ref_st == 1
    n, _, _ = check(case)
    assert n == case.T - 3   # T = 4 x 32 = 128 tokens fill the 128 slots; 3 are bad


def test_all_skipped_and_empty():
    case = wl.make_kv_case("e", 3, 5, mode="PA_BSND", d0=2, d1=16, seed=50)
    case.index[:] = -1
    n, _, _ = check(case)
    assert n == 0
    case = wl.make_kv_case("e", 0, 5, mode="PA_BSND", d0=2, d1=16, seed=50)
    g_ckv, g_k, st = run_gpu_kv(case)
    assert st == 0 and np.all(g_ckv == wl.SENTINEL16) and np.all(g_k == wl.SENTINEL16)


def test_norm_mode_with_larger_cache_batch_and_shared_slots():
    """Norm indices may repeat across batches: each batch owns its cache row."""
    case = wl.make_kv_case("n", 3, 10, mode="Norm", d0=5, d1=10, seed=51)
    case.index[:] = torch.arange(10).flip(0)
    check(case)


def test_repeated_calls_overwrite_only_their_rows():
    """Two calls into the same caches: the second overwrites its own rows only."""
    a = wl.make_kv_case("c", 4, 16, mode="PA_BSND", d0=16, d1=16, seed=52)
    b = wl.make_kv_case("c", 4, 16, mode="PA_BSND", d0=16, d1=16, seed=53)
    ckv = sentinel_cache((16, 16, 1, 512), "bf16")
    k = sentinel_cache((16, 16, 1, 64), "bf16")
    run_gpu_kv(a, ckv=ckv, k=k)
    g_ckv, g_k, st = run_gpu_kv(b, ckv=ckv, k=k)
    r_ckv, r_k, _ = run_oracle_kv(a)
    run_oracle_kv(b, r_ckv, r_k)
    compare_cache(g_ckv, r_ckv, "bf16", 512)
    compare_cache(g_k, r_k, "bf16", 64)


def test_large_ragged_grid_stride():
    """More rows than the grid holds at once, with a ragged tail."""
    case = wl.make_kv_case("g", 3, 9001, mode="PA_BSND", d0=300, d1=128, seed=54, skip=101)
    check(case)


BULK_CASES = {
    # (Bkv, Skv, make_kv_case keywords): every case has >= 8192 rows (the pipeline kernel)
    "threshold_8192": (1, 8192, dict(mode="PA_BSND", d0=80, d1=128, skip=17)),
    "odd_8193": (1, 8193, dict(mode="PA_BSND", d0=80, d1=128, skip=3)),
    "norm_odd": (3, 6667, dict(mode="Norm", d0=4, d1=6700, skip=11)),
    "blk_bsnd": (5, 2000, dict(mode="PA_BLK_BSND", d0=5 * 16 + 3, d1=128)),
    "fp8_per_channel": (2, 5003, dict(mode="PA_BSND", d0=100, d1=128, ckv_dtype="fp8_e4m3fn", kv_std=3.0)),
    "int8_e5m2_per_tensor": (2, 4500, dict(mode="PA_BSND", d0=80, d1=128, ckv_dtype="int8", k_dtype="fp8_e5m2",
                                            scale_len=1, k_scale_len=1, kv_std=3.0)),
    "strided_rows": (4, 2500, dict(mode="PA_BSND", d0=90, d1=128, row_pad=64, skip=9)),
    "f16": (2, 4200, dict(mode="PA_BSND", d0=80, d1=128, in_dtype="f16", ckv_dtype="f16", k_dtype="f16")),
    "other_split": (2, 4600, dict(mode="PA_BSND", Dv=256, Dk=32, d0=80, d1=128, skip=5)),
}


@pytest.mark.parametrize("name", sorted(BULK_CASES))
def test_bulk_pipeline_paths(name):
    """The bulk-copy pipeline (batches of 8192 rows or more): each SM's row
    range, ragged last tiles, per-row copies of strided rows, index entries
    read from global memory (PA_BLK_BSND), 8-bit codes, f16 and another row
    split, against the oracle."""
    Bkv, Skv, kw = BULK_CASES[name]
    case = wl.make_kv_case("bulk_" + name, Bkv, Skv, seed=7000 + len(name), **kw)
    assert case.T >= 8192
    n, _, _ = check(case)
    assert n == case.active_tokens()


def test_bulk_pipeline_misaligned_index_and_bad_entries():
    """An index buffer at an 8-byte (not 16-byte) offset takes the global
    index reads; out-of-range entries are skipped and flagged."""
    import attention_prologue_kv_gb300 as kvr
    case = wl.make_kv_case("bulk_idx", 2, 4800, mode="PA_BSND", d0=80, d1=128, seed=7100, skip=7)
    case.index[5] = 80 * 128
    case.index[9000] = -3
    ref_ckv, ref_k, ref_st = run_oracle_kv(case)
    assert ref_st == 1
    buf = torch.empty(case.T + 1, dtype=torch.int64, device="cuda")
    idx = buf[1:]
    idx.copy_(case.index)
    assert idx.data_ptr() % 16 == 8
    ckv, c1 = guarded_cache(case.cache_shapes()[0], "bf16")
    k, c2 = guarded_cache(case.cache_shapes()[1], "bf16")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvr.kv_rmsnorm_rope_cache(case.kv.cuda(), case.gamma.cuda(), case.cos.cuda(), case.sin.cuda(), idx, ckv, k,
                              cache_mode="PA_BSND", eps=case.eps, dev_status=status)
    torch.cuda.synchronize()
    c1()
    c2()
    assert int(status.item()) == ref_st
    n1, _ = compare_cache(codes_of(ckv), ref_ckv, "bf16", case.Dv)
    n2, _ = compare_cache(codes_of(k), ref_k, "bf16", case.Dk)
    assert n1 == n2 == case.active_tokens() - 2


def test_rope_identity_on_gpu_is_exact_deinterleave():
    case = wl.make_kv_case("i", 2, 8, mode="PA_BSND", d0=1, d1=16, seed=55)
    case.cos[:] = 1.0
    case.sin[:] = 0.0
    _, g_k, _ = run_gpu_kv(case)
    x = case.kv.reshape(-1, 576)[:, 512:].view(torch.int16).numpy().view(np.uint16)
    want = np.concatenate([x[:, 0::2], x[:, 1::2]], axis=1)
    assert np.array_equal(g_k.reshape(-1, 64)[case.index.numpy()], want)


def test_prepared_call_matches_the_plain_call_and_sees_new_contents():
    """A prepared call bound to fixed buffers: refilling the buffers between
    calls gives each batch's own result."""
    import attention_prologue_kv_gb300 as kvr
    a = wl.make_kv_case("p", 4, 16, mode="PA_BSND", d0=16, d1=16, seed=60, skip=3)
    b = wl.make_kv_case("p", 4, 16, mode="PA_BSND", d0=16, d1=16, seed=61, skip=2)
    kv, cos, sin, idx = (a.kv.cuda(), a.cos.cuda(), a.sin.cuda(), a.index.cuda())
    ckv = sentinel_cache((16, 16, 1, 512), "bf16")
    k = sentinel_cache((16, 16, 1, 64), "bf16")
    call = kvr.prepare_kv_rmsnorm_rope_cache(kv, a.gamma.cuda(), cos, sin, idx, ckv, k, cache_mode="PA_BSND")
    call()
    kv.copy_(b.kv)
    cos.copy_(b.cos)
    sin.copy_(b.sin)
    idx.copy_(b.index)
    b.gamma = a.gamma
    call()
    torch.cuda.synchronize()
    r_ckv, r_k, _ = run_oracle_kv(a)
    run_oracle_kv(b, r_ckv, r_k)
    from helpers import codes_of
    compare_cache(codes_of(ckv), r_ckv, "bf16", 512)
    compare_cache(codes_of(k), r_k, "bf16", 64)


@pytest.mark.parametrize("make", [
    wl.decode_paged, wl.quant_fp8,
    lambda: wl.make_kv_case("p", 8, 40, mode="PA_BSND", d0=8, d1=64, ckv_dtype="int8", k_dtype="fp8_e4m3fn",
                            seed=64, skip=3, kv_std=3.0, scale_len=1),
    lambda: wl.make_kv_case("p", 8, 40, mode="PA_BSND", d0=8, d1=64, ckv_dtype="fp8_e5m2", k_dtype="int8",
                            seed=65, kv_std=3.0),
    lambda: wl.make_kv_case("p", 4, 9, Dv=20, Dk=6, mode="PA_BSND", d0=4, d1=16, ckv_dtype="fp8_e4m3fn",
                            k_dtype="int8", seed=66)],
    ids=["decode_paged", "quant_fp8", "per_tensor_scales", "per_channel_k_scale", "generic_path"])
def test_params_ready_gives_the_same_result(make):
    """params_ready only moves the reads of gamma and the scales before the
    dependency wait: the register flavour (decode), the shared-memory flavour
    (quant), per-tensor and per-channel scales, and the generic path agree
    with the oracle as without it."""
    case = make()
    check(case, params_ready=True)


def test_staged_call_from_pinned_host_memory():
    """kv_rmsnorm_rope_cache_staged: two batches staged from pinned host
    memory into one device buffer, each followed by its call and a status
    read-back; the caches equal the oracle's after both batches, the status
    words arrive on the host (0 for a valid batch, the index bit for one with
    an out-of-range slot), and a call with host tensors checks them."""
    import attention_prologue_kv_gb300 as kvr
    from helpers import codes_of
    a = wl.make_kv_case("s", 4, 16, mode="PA_BSND", d0=16, d1=16, seed=62, skip=3)
    b = wl.make_kv_case("s", 4, 16, mode="PA_BSND", d0=16, d1=16, seed=63, skip=2)
    b.index[5] = 16 * 16 + 7     # out of range: skipped, KVR_DEVERR_INDEX
    parts = lambda c: [c.kv.reshape(-1).view(torch.uint8), c.cos.reshape(-1).view(torch.uint8),
                       c.sin.reshape(-1).view(torch.uint8), c.index.reshape(-1).view(torch.uint8)]
    sizes = [t.numel() for t in parts(a)]
    blob = sum(sizes)
    host = torch.empty(2, blob, dtype=torch.uint8).pin_memory()
    for r, c in enumerate((a, b)):
        host[r] = torch.cat(parts(c))
    stage = torch.zeros(blob, dtype=torch.uint8, device="cuda")
    o = [0]
    for n in sizes:
        o.append(o[-1] + n)
    kv = stage[o[0]:o[1]].view(torch.bfloat16).view(a.kv.shape)
    cos = stage[o[1]:o[2]].view(torch.bfloat16).view(a.cos.shape)
    sin = stage[o[2]:o[3]].view(torch.bfloat16).view(a.sin.shape)
    idx = stage[o[3]:o[4]].view(torch.int64)
    ckv = sentinel_cache((16, 16, 1, 512), "bf16")
    k = sentinel_cache((16, 16, 1, 64), "bf16")
    dev_status = torch.zeros(1, dtype=torch.int32, device="cuda")
    host_status = torch.full((2,), -1, dtype=torch.int32).pin_memory()
    call = kvr.prepare_kv_rmsnorm_rope_cache(kv, a.gamma.cuda(), cos, sin, idx, ckv, k, cache_mode="PA_BSND",
                                             dev_status=dev_status)
    call.staged(host[0], stage, blob, host_status[0:1])
    call.staged(host[1].data_ptr(), stage.data_ptr(), blob, host_status[1:2].data_ptr())
    torch.cuda.synchronize()
    assert host_status.tolist() == [0, 0x1]
    b.gamma = a.gamma
    r_ckv, r_k, _ = run_oracle_kv(a)
    run_oracle_kv(b, r_ckv, r_k)
    compare_cache(codes_of(ckv), r_ckv, "bf16", 512)
    compare_cache(codes_of(k), r_k, "bf16", 64)
    with pytest.raises(ValueError):
        call.staged(host[0].clone(), stage, blob)          # not pinned
    # pageable memory by raw address: staged through a copy-engine operation
    pageable = host[1].clone().numpy()
    ckv.view(torch.int16).fill_(wl.SENTINEL16)
    k.view(torch.int16).fill_(wl.SENTINEL16)
    dev_status.zero_()
    call.staged(pageable.ctypes.data, stage.data_ptr(), blob, host_status[0:1].data_ptr())
    torch.cuda.synchronize()
    assert int(host_status[0]) == 0x1
    r_ckv2, r_k2, _ = run_oracle_kv(b)
    compare_cache(codes_of(ckv), r_ckv2, "bf16", 512)
    compare_cache(codes_of(k), r_k2, "bf16", 64)


def test_staged_large_batch():
    """A 5.8 MB staged input (4096 tokens): more 16-byte elements than the
    copy kernel has threads, so its grid-stride loop runs several rounds;
    three steps in a row through one staging buffer."""
    import attention_prologue_kv_gb300 as kvr
    from helpers import codes_of
    cases = [wl.make_kv_case("sl", 64, 64, mode="PA_BSND", d0=512, d1=128, seed=70 + i, skip=9) for i in range(3)]
    parts = lambda c: [c.kv.reshape(-1).view(torch.uint8), c.cos.reshape(-1).view(torch.uint8),
                       c.sin.reshape(-1).view(torch.uint8), c.index.reshape(-1).view(torch.uint8)]
    sizes = [t.numel() for t in parts(cases[0])]
    blob = sum(sizes)
    assert blob // 16 > 4 * 304 * 256
    host = torch.empty(len(cases), blob, dtype=torch.uint8).pin_memory()
    for r, c in enumerate(cases):
        host[r] = torch.cat(parts(c))
    stage = torch.zeros(blob, dtype=torch.uint8, device="cuda")
    o = [0]
    for n in sizes:
        o.append(o[-1] + n)
    c0 = cases[0]
    views = (stage[o[0]:o[1]].view(torch.bfloat16).view(c0.kv.shape),
             stage[o[1]:o[2]].view(torch.bfloat16).view(c0.cos.shape),
             stage[o[2]:o[3]].view(torch.bfloat16).view(c0.sin.shape), stage[o[3]:o[4]].view(torch.int64))
    ckv = sentinel_cache((512, 128, 1, 512), "bf16")
    k = sentinel_cache((512, 128, 1, 64), "bf16")
    call = kvr.prepare_kv_rmsnorm_rope_cache(views[0], c0.gamma.cuda(), views[1], views[2], views[3], ckv, k,
                                             cache_mode="PA_BSND")
    for r in range(len(cases)):
        call.staged(host[r], stage, blob)
    torch.cuda.synchronize()
    r_ckv = r_k = None
    for c in cases:
        c.gamma = c0.gamma
        r_ckv, r_k, _ = run_oracle_kv(c, r_ckv, r_k) if r_ckv is not None else run_oracle_kv(c)
    compare_cache(codes_of(ckv), r_ckv, "bf16", 512)
    compare_cache(codes_of(k), r_k, "bf16", 64)


def test_benchmark_decode_sets_match_the_oracle():
    """The rotating decode batches the benchmark times, through the same
    call and launch configuration, against the oracle (first four sets)."""
    import attention_prologue_kv_gb300 as kvr
    import oracle
    from helpers import codes_of
    sets = wl.decode_paged_sets(4)
    d0, d1 = sets["d0"], sets["d1"]
    ckv = sentinel_cache((d0, d1, 1, 512), "bf16")
    k = sentinel_cache((d0, d1, 1, 64), "bf16")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    r_ckv = np.full((d0, d1, 512), wl.SENTINEL16, dtype=np.uint16)
    r_k = np.full((d0, d1, 64), wl.SENTINEL16, dtype=np.uint16)
    g = sets["gamma"].cuda()
    for i in range(4):
        kvr.kv_rmsnorm_rope_cache(sets["kv"][i].cuda(), g, sets["cos"][i].cuda(), sets["sin"][i].cuda(),
                                  sets["index"][i].cuda(), ckv, k, cache_mode="PA_BSND", dev_status=st)
        oracle.ref_kv_rmsnorm_rope_cache(
            sets["kv"][i].double().numpy().reshape(-1, 1, 576), sets["gamma"].double().numpy(),
            sets["cos"][i].double().numpy().reshape(-1, 1, 64), sets["sin"][i].double().numpy().reshape(-1, 1, 64),
            sets["index"][i].numpy(), r_ckv, r_k, Dv=512, mode="PA_BSND", eps=1e-6)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    n, _ = compare_cache(codes_of(ckv), r_ckv, "bf16", 512)
    assert n == 4 * 251
    compare_cache(codes_of(k), r_k, "bf16", 64)
