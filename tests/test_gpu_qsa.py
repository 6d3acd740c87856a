"""GPU parity of qsa_prepare against the float64 oracle: block keys within
2**-7*|ref| + 1e-6, untouched block rows bit-exact, carry outputs bit-exact
(they are copies), device status bits equal; chained calls through the carry
outputs equal one call."""
import numpy as np
import pytest
import torch

from attention_prologue_kv_gb300 import workloads as wl
from helpers import check_robust_qsa, compare_cache, run_gpu_qsa, run_oracle_qsa

pytestmark = pytest.mark.gpu


def check(case, carry=True, rope_layout="interleave_last", past_block_keys=None, params_ready=False,
          late_key_length=None, key_length_late=False):
    kw = dict(carry=carry, rope_layout=rope_layout, past_block_keys=past_block_keys)
    values = {}
    r_bk, r_nr, r_npr, r_st = run_oracle_qsa(case, values_out=values, **kw)
    g_bk, g_nr, g_npr, g_st = run_gpu_qsa(case, params_ready=params_ready, late_key_length=late_key_length,
                                          key_length_late=key_length_late, **kw)
    assert g_st == r_st
    if past_block_keys is not None:
        # copied past rows are bit-exact copies
        for n, P in enumerate(case.meta["past"]):
            m = min(past_block_keys.shape[1], P // case.kbs, case.Bcap)
            assert np.array_equal(g_bk[n, :m], r_bk[n, :m])
    dt = "f16" if case.raw.dtype == torch.float16 else "bf16"
    n, exact = compare_cache(g_bk, r_bk, dt, case.Di)
    check_robust_qsa(g_bk, values, dt)
    if carry:
        assert np.array_equal(g_nr, r_nr, equal_nan=True)
        if case.Dr:
            assert np.array_equal(g_npr, r_npr, equal_nan=True)
    return n, exact


def test_workload_full_size():
    case = wl.qsa_prepare_workload()
    n, exact = check(case)
    assert n == 32 * 32 == case.completed_blocks()
    assert exact > 0.97


@pytest.mark.parametrize("Di,Dr,kbs", [(128, 64, 64), (24, 8, 5), (16, 16, 2), (12, 4, 3),
                                       (2048, 64, 16), (4096, 128, 4), (4000, 0, 7), (8, 2, 64)])
def test_shapes(Di, Dr, kbs):
    case = wl.make_qsa_case("s", 5, 37, Di=Di, Dr=Dr, kbs=kbs, seed=Di + kbs, past_max=300,
                            rope=Dr > 0)
    check(case)


@pytest.mark.parametrize("rope,norm", [(False, False), (False, True), (True, False)])
def test_features_disabled(rope, norm):
    case = wl.make_qsa_case("f", 6, 50, Di=32, Dr=8, kbs=4, seed=7, rope=rope, norm=norm)
    check(case)


def test_shared_key_length():
    case = wl.make_qsa_case("k", 4, 33, Di=64, Dr=16, kbs=8, seed=8, shared_length=True)
    check(case)


def stale_key_lengths(case, late):
    K = case.key_length
    return {"same": K.clone(), "one_block_more": K + case.kbs, "ragged_less": (K - 17).clamp(min=0),
            "below_L": torch.full_like(K, case.L - 1), "huge": torch.full_like(K, 1 << 62),
            "mixed": torch.where(torch.arange(K.numel()) % 2 == 0, K + 3, K)}[late]


@pytest.mark.parametrize("flag", [False, True])
@pytest.mark.parametrize("late", ["same", "one_block_more", "ragged_less", "below_L", "huge", "mixed"])
@pytest.mark.parametrize("L,Di,kbs,shared", [(2048, 128, 64, False), (300, 64, 32, True), (45, 256, 128, False)])
def test_key_length_written_late_by_the_preceding_kernel(late, L, Di, kbs, shared, flag):
    """The default form reads key_length before its dependency wait only as
    a prefetch hint. Here the kernel launched just before the call lets it
    start and writes key_length afterwards; the call still finds the blocks,
    carry outputs and status of the late values, whatever the stale ones
    were: the same, a block further on, a ragged amount less, shorter than L
    (no usable hint), huge (blocks beyond Bcap), or stale in every other
    sequence only; with and without key_length_late (no hint taken)."""
    case = wl.make_qsa_case("late", 8, L, Di=Di, Dr=64, kbs=kbs, seed=L + Di + kbs, past_max=4 * kbs + 7,
                            shared_length=shared)
    n, _ = check(case, late_key_length=stale_key_lengths(case, late), key_length_late=flag)
    assert n == case.completed_blocks()


@pytest.mark.parametrize("flag", [False, True])
@pytest.mark.parametrize("late", ["one_block_more", "mixed"])
def test_key_length_written_late_full_size(late, flag):
    """The benchmark's workload (32 sequences of 2048 new tokens, per-sequence
    key_length) with its key lengths written after the call has started."""
    case = wl.qsa_prepare_workload()
    n, _ = check(case, late_key_length=stale_key_lengths(case, late), key_length_late=flag)
    assert n == case.completed_blocks() == 1024


def test_key_length_late_flag_without_a_late_write():
    """key_length_late only drops the hint: with key_length written well
    before the call the results are the same, full size and with carry."""
    case = wl.qsa_prepare_workload()
    n, _ = check(case, key_length_late=True)
    assert n == 1024


def test_no_block_completed_only_carry():
    case = wl.make_qsa_case("c", 3, 3, Di=32, Dr=8, kbs=16, seed=9, past=[0, 5, 12])
    n, _ = check(case)
    # key lengths 3, 8, 15 with kbs 16: no block completes; only the carry outputs change
    assert n == case.completed_blocks() == 0


def test_device_status_bits():
    case = wl.make_qsa_case("e", 3, 16, Di=16, Dr=8, kbs=4, seed=10, past=[0, 3, 40], Bcap=12)
    case.key_length = torch.tensor([10, 19, 56])   # sequence 0: key_length < L; sequence 2: blocks >= Bcap
    r_bk, _, _, r_st = run_oracle_qsa(case)
    assert r_st == 0x2 | 0x4
    check(case)


def test_chained_calls_on_gpu_equal_one_call():
    N, L, Di, Dr, kbs = 4, 45, 32, 8, 6
    case = wl.make_qsa_case("t", N, L, Di=Di, Dr=Dr, kbs=kbs, seed=11, past=[0, 5, 13, 6], Bcap=12)
    whole, _, _, _ = run_gpu_qsa(case, carry=False)
    import attention_prologue_kv_gb300 as kvr
    dev = "cuda"
    bk = torch.full((N, 12, Di), wl.SENTINEL16, dtype=torch.int16, device=dev).view(torch.bfloat16)
    past_raw, past_rope = case.past_raw.to(dev), case.past_rope.to(dev)
    P = torch.tensor(case.meta["past"])
    for a, b in [(0, 7), (7, 30), (30, L)]:
        nr = torch.full((N, kbs - 1, Di), float("nan"), dtype=torch.bfloat16, device=dev)
        npr = torch.full((N, 2 * Dr), float("nan"), dtype=torch.bfloat16, device=dev)
        kvr.qsa_prepare(case.raw[:, a:b].contiguous().to(dev), bk, (P + b).to(dev),
                        case.rope_cos[:, a:b].contiguous().to(dev), case.rope_sin[:, a:b].contiguous().to(dev),
                        case.k_norm_weight.to(dev), past_raw, past_rope, kbs, case.eps,
                        next_incomplete_raw_keys=nr, next_incomplete_rope=npr)
        past_raw, past_rope = nr, npr
    torch.cuda.synchronize()
    assert np.array_equal(bk.cpu().view(torch.int16).numpy(), whole.view(np.int16))


def test_empty():
    case = wl.make_qsa_case("z", 3, 0, Di=32, Dr=8, kbs=4, seed=12)
    g_bk, _, _, st = run_gpu_qsa(case)
    assert st == 0 and np.all(g_bk == wl.SENTINEL16)


@pytest.mark.parametrize("N,L,Di,Dr,kbs", [(3, 600, 128, 64, 128), (40, 300, 64, 16, 8)])
def test_pipeline_ring_depths(N, L, Di, Dr, kbs):
    """Shapes whose blocks go through a 4-stage ring (kbs = 128) and through an
    8-stage ring with many blocks per CTA (the ring wraps many times)."""
    case = wl.make_qsa_case("r", N, L, Di=Di, Dr=Dr, kbs=kbs, seed=N + L, past_max=500)
    n, _ = check(case)
    assert n == case.completed_blocks()


# ---- RoPE layouts on each kernel variant: one warp per block (Di, kbs
# compiled: 128, 64), bulk copies (Di, Dr multiples of 8, other kbs: 128, 64,
# 5 and 16, 16, 2), register loads (Dr not a multiple of 8), scalar loads (Di
# odd multiple of 4) ----

@pytest.mark.parametrize("layout", ["interleave_last", "interleave_first", "half_last", "half_first"])
@pytest.mark.parametrize("Di,Dr,kbs", [(128, 64, 64), (128, 64, 5), (24, 6, 5), (12, 4, 3), (16, 16, 2)])
def test_rope_layouts(layout, Di, Dr, kbs):
    case = wl.make_qsa_case("l", 5, 37, Di=Di, Dr=Dr, kbs=kbs, seed=Di * 3 + kbs, past_max=300)
    n, _ = check(case, rope_layout=layout)
    assert n == case.completed_blocks()


def test_rope_layout_full_size_half_first():
    case = wl.qsa_prepare_workload()
    n, exact = check(case, rope_layout="half_first")
    assert n == case.completed_blocks() and exact > 0.97


# ---- concat-output form ----

def _past_codes(case, Bp, seed):
    return np.random.default_rng(seed).integers(0, 0x7F00, (case.N, Bp, case.Di), dtype=np.uint16)


def test_concat_form_full_size():
    case = wl.qsa_prepare_workload()
    P = np.array(case.meta["past"])
    past = _past_codes(case, int((P // case.kbs).max()), 31)
    n, exact = check(case, past_block_keys=past)
    assert n == case.completed_blocks() + int((P // case.kbs).sum())


@pytest.mark.parametrize("Di,Dr,kbs", [(128, 64, 4), (24, 8, 3), (12, 4, 2), (8192 // 2, 64, 2)])
def test_concat_form_shapes(Di, Dr, kbs):
    """Several copy CTAs per sequence (Di = 128, 4096: 64 rows and 2 rows per
    CTA), the 16-byte and the 2-byte copy."""
    case = wl.make_qsa_case("c", 4, 21, Di=Di, Dr=Dr, kbs=kbs, seed=Di + kbs, past_max=400)
    P = np.array(case.meta["past"])
    past = _past_codes(case, int((P // kbs).max()) + 3, Di)
    check(case, past_block_keys=past)


def test_concat_form_status_bits():
    # sequence 1: 5 past blocks but a 3-row past buffer; sequence 2: past rows beyond Bcap
    case = wl.make_qsa_case("s", 3, 4, Di=16, Dr=8, kbs=4, seed=32, past=[4, 20, 40], Bcap=9)
    past = _past_codes(case, 3, 33)
    assert run_oracle_qsa(case, past_block_keys=past)[3] == 0x10 | 0x4
    check(case, past_block_keys=past)
    case2 = wl.make_qsa_case("s", 1, 4, Di=16, Dr=8, kbs=4, seed=34, past=[40], Bcap=6)
    past2 = _past_codes(case2, 12, 35)
    assert run_oracle_qsa(case2, past_block_keys=past2)[3] == 0x4
    check(case2, past_block_keys=past2)


def test_concat_form_same_buffer_is_in_place():
    import attention_prologue_kv_gb300 as kvr
    case = wl.make_qsa_case("i", 3, 20, Di=32, Dr=8, kbs=4, seed=36, past=[0, 6, 13])
    ref, _, _, _ = run_gpu_qsa(case)
    dev = "cuda"
    bk = torch.full((case.N, case.Bcap, case.Di), wl.SENTINEL16, dtype=torch.int16, device=dev).view(torch.bfloat16)
    d = lambda t: t.to(dev)
    kvr.qsa_prepare(d(case.raw), bk, d(case.key_length), d(case.rope_cos), d(case.rope_sin),
                    d(case.k_norm_weight), d(case.past_raw), d(case.past_rope), case.kbs, case.eps,
                    past_block_index_keys=bk)
    torch.cuda.synchronize()
    assert np.array_equal(bk.cpu().view(torch.int16).numpy(), ref.view(np.int16))


def test_no_new_tokens_still_writes_carry_and_past_rows():
    """L = 0: no block completes, but the carry outputs pass the carried keys
    on and the concat form still copies the past rows."""
    case = wl.make_qsa_case("z", 3, 0, Di=32, Dr=8, kbs=4, seed=37, past=[5, 8, 14])
    P = np.array(case.meta["past"])
    n, _ = check(case, carry=True, past_block_keys=_past_codes(case, 4, 38))
    assert n == int(np.minimum(P // 4, 4).sum())


def test_chained_concat_calls_equal_one_call():
    """Each call writes a fresh buffer from the previous one (concat form);
    the last equals one in-place call over all tokens."""
    import attention_prologue_kv_gb300 as kvr
    N, L, Di, Dr, kbs = 3, 40, 32, 8, 6
    case = wl.make_qsa_case("t", N, L, Di=Di, Dr=Dr, kbs=kbs, seed=39, past=[0, 5, 13], Bcap=12)
    whole, _, _, _ = run_gpu_qsa(case, carry=False)
    dev = "cuda"
    P = torch.tensor(case.meta["past"])
    prev = torch.full((N, 12, Di), wl.SENTINEL16, dtype=torch.int16, device=dev).view(torch.bfloat16)
    past_raw, past_rope = case.past_raw.to(dev), case.past_rope.to(dev)
    for a, b in [(0, 9), (9, 25), (25, L)]:
        out = torch.full((N, 12, Di), wl.SENTINEL16, dtype=torch.int16, device=dev).view(torch.bfloat16)
        nr = torch.full((N, kbs - 1, Di), float("nan"), dtype=torch.bfloat16, device=dev)
        npr = torch.full((N, 2 * Dr), float("nan"), dtype=torch.bfloat16, device=dev)
        kvr.qsa_prepare(case.raw[:, a:b].contiguous().to(dev), out, (P + b).to(dev),
                        case.rope_cos[:, a:b].contiguous().to(dev), case.rope_sin[:, a:b].contiguous().to(dev),
                        case.k_norm_weight.to(dev), past_raw, past_rope, kbs, case.eps,
                        next_incomplete_raw_keys=nr, next_incomplete_rope=npr, past_block_index_keys=prev)
        prev, past_raw, past_rope = out, nr, npr
    torch.cuda.synchronize()
    assert np.array_equal(prev.cpu().view(torch.int16).numpy(), whole.view(np.int16))


def test_buffer_lengths_are_checked():
    """Tables, weights and carry buffers of the wrong length are refused
    before launch (the C ABI cannot see a buffer's length)."""
    import attention_prologue_kv_gb300 as kvr
    case = wl.make_qsa_case("b", 3, 20, Di=32, Dr=8, kbs=4, seed=40)
    d = lambda t: t.cuda()
    bk = torch.zeros(3, case.Bcap, 32, dtype=torch.bfloat16, device="cuda")
    args = [d(case.raw), bk, d(case.key_length), d(case.rope_cos), d(case.rope_sin), d(case.k_norm_weight),
            d(case.past_raw), d(case.past_rope), case.kbs]
    for pos, short in ((3, d(case.rope_cos[:, :10]).contiguous()), (5, d(case.k_norm_weight[:16])),
                       (6, d(case.past_raw[:2])), (7, d(case.past_rope[:, :8]).contiguous())):
        bad = list(args)
        bad[pos] = short
        with pytest.raises(ValueError):
            kvr.qsa_prepare(*bad)
    with pytest.raises(ValueError):
        kvr.qsa_prepare(*args, next_incomplete_raw_keys=torch.zeros(3, 2, 32, dtype=torch.bfloat16, device="cuda"))
    kvr.qsa_prepare(*args)   # the well-formed call still runs
    torch.cuda.synchronize()


@pytest.mark.parametrize("Di", [64, 128, 256])
@pytest.mark.parametrize("kbs", [32, 64, 128])
def test_compile_time_shapes(Di, kbs):
    """The kernels compiled for fixed (Di, kbs) pairs, with the carry outputs
    and a RoPE layout that changes from case to case."""
    layout = ["interleave_last", "half_first", "interleave_first", "half_last"][(Di // 64 + kbs // 32) % 4]
    case = wl.make_qsa_case("sp", 4, 300, Di=Di, Dr=min(64, Di), kbs=kbs, seed=Di + kbs, past_max=600)
    n, _ = check(case, rope_layout=layout)
    assert n == case.completed_blocks()


@pytest.mark.parametrize("rope,norm", [(False, True), (True, False)])
def test_compile_time_shape_features_disabled(rope, norm):
    case = wl.make_qsa_case("sp", 5, 200, Di=128, Dr=64, kbs=64, seed=77, rope=rope, norm=norm, past_max=500)
    check(case)


def test_compile_time_shape_concat_form():
    case = wl.make_qsa_case("sp", 6, 256, Di=128, Dr=64, kbs=32, seed=78, past_max=700)
    P = np.array(case.meta["past"])
    check(case, past_block_keys=_past_codes(case, int((P // 32).max()) + 2, 79))


def test_concat_form_with_an_empty_past_buffer():
    """Bp = 0 is still the concat-output form: every sequence with past
    blocks raises KVR_DEVERR_PAST_BLOCKS (an empty tensor has no address,
    which the C call would otherwise read as in place)."""
    case = wl.make_qsa_case("e", 3, 40, Di=128, Dr=64, kbs=32, seed=80, past=[0, 40, 70])
    past = np.zeros((3, 0, 128), dtype=np.uint16)
    assert run_oracle_qsa(case, past_block_keys=past)[3] == 0x10
    check(case, past_block_keys=past)


@pytest.mark.parametrize("Di,kbs", [(64, 128), (128, 64), (256, 32)])
def test_params_ready(Di, kbs):
    """params_ready: the compiled-shape kernel reads key_length, the tables
    and the weight before its dependency wait; results are unchanged (carry
    outputs on, every RoPE layout family)."""
    layout = {64: "half_first", 128: "interleave_last", 256: "interleave_first"}[Di]
    case = wl.make_qsa_case("pr", 5, 333, Di=Di, Dr=min(64, Di), kbs=kbs, seed=Di + kbs + 1, past_max=900)
    n, _ = check(case, rope_layout=layout, params_ready=True)
    assert n == case.completed_blocks()


def test_params_ready_full_size_and_status():
    """The workload with params_ready, then a case whose key_length is short
    of L for one sequence and whose blocks overflow Bcap for another: the
    status bits are raised after the wait exactly as without the flag."""
    case = wl.qsa_prepare_workload()
    n, exact = check(case, params_ready=True)
    assert n == 32 * 32 and exact > 0.97
    bad = wl.make_qsa_case("prs", 3, 256, Di=128, Dr=64, kbs=64, seed=91, past=[0, 70, 300], Bcap=6)
    bad.key_length[0] = 100     # < L: KVR_DEVERR_KEY_LENGTH, sequence skipped
    assert run_oracle_qsa(bad)[3] == 0x2 | 0x4
    for ready in (False, True):
        check(bad, params_ready=ready)   # status bits equal to the oracle's


def test_params_ready_concat_form():
    case = wl.make_qsa_case("prc", 6, 256, Di=128, Dr=64, kbs=64, seed=92, past_max=2000)
    P = np.array(case.meta["past"])
    check(case, past_block_keys=_past_codes(case, int((P // 64).max()) + 1, 93), params_ready=True)


def test_compiled_shape_unaligned_buffers():
    """The warp kernel's 2-byte paths: carry outputs and past block keys that
    start 2 bytes past a 16-byte boundary (the block keys stay aligned)."""
    import attention_prologue_kv_gb300 as kvr
    from helpers import codes_of, f64
    case = wl.make_qsa_case("ua", 3, 200, Di=128, Dr=64, kbs=64, seed=95, past=[10, 130, 300])
    P = np.array(case.meta["past"])
    past = _past_codes(case, int((P // 64).max()) + 1, 96)
    r_bk, r_nr, r_npr, r_st = run_oracle_qsa(case, carry=True, past_block_keys=past)
    dev, dt = "cuda", case.raw.dtype

    def off_by_one(codes):
        flat = torch.from_numpy(np.ascontiguousarray(codes).view(np.int16).reshape(-1)).to(dev)
        buf = torch.zeros(flat.numel() + 1, dtype=torch.int16, device=dev)
        buf[1:] = flat
        return buf[1:].view(dt).view(codes.shape)

    nan_codes = np.full((case.N, 63, 128), 0x7FC0, dtype=np.uint16)
    nr = off_by_one(nan_codes)
    assert nr.data_ptr() % 16 == 2
    pbk = off_by_one(past)
    npr = torch.full((case.N, 128), float("nan"), dtype=dt, device=dev)
    bk = torch.full((case.N, case.Bcap, 128), 0x7FBF, dtype=torch.int16, device=dev).view(dt)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    d = lambda t: t.to(dev)
    for ready in (False, True):
        kvr.qsa_prepare(d(case.raw), bk, d(case.key_length), d(case.rope_cos), d(case.rope_sin),
                        d(case.k_norm_weight), d(case.past_raw), d(case.past_rope), 64, case.eps,
                        next_incomplete_raw_keys=nr, next_incomplete_rope=npr, dev_status=st,
                        past_block_index_keys=pbk, params_ready=ready)
        torch.cuda.synchronize()
        assert int(st.item()) == r_st
        compare_cache(codes_of(bk), r_bk, "bf16", 128)
        assert np.array_equal(f64(nr), r_nr, equal_nan=True)
        assert np.array_equal(f64(npr), r_npr, equal_nan=True)


@pytest.mark.parametrize("params_ready", [False, True])
def test_f16_full_size(params_ready):
    """The workload's shape with f16 keys, weight and tables (the output type
    follows the input), in both forms, with carry outputs."""
    case = wl.make_qsa_case("qsa_f16", 32, 2048, Di=128, Dr=64, kbs=64, seed=1205, past_max=8192, Bcap=160,
                            in_dtype="f16")
    n, _ = check(case, params_ready=params_ready)
    assert n == case.completed_blocks()
