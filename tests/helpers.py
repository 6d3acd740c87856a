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


def f32_arg(x):
    """The value a float argument of the C call holds (it is passed as a
    C float): what the oracle must be given for the same call."""
    return float(np.float32(x))


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
    st = fn(kv, gamma, cos, sin, index, ckv, k, Dv=case.Dv, mode=case.mode, eps=f32_arg(case.eps),
            ckv_dtype=case.ckv_dtype, k_dtype=case.k_dtype,
            ckv_scale=None if case.ckv_scale is None else case.ckv_scale.numpy(),
            k_scale=None if case.k_scale is None else case.k_scale.numpy(),
            kc_scale=f32_arg(case.kc_scale))
    return ckv, k, st


ROBUST_REL = 2.0 ** -17   # perturbation within which a float32 evaluation may land on either side


def robust_codes(v, margin, dtype):
    """(codes of v, mask): the mask marks elements whose code does not change
    anywhere in [v - margin, v + margin] (the encoders are monotone, so the
    ends decide), i.e. elements no evaluation within that error can round
    differently."""
    from oracle import encoders as enc
    want = enc.encode(v, dtype)
    return want, enc.encode(v - margin, dtype) == enc.encode(v + margin, dtype)


def kv_token_rows(case):
    """Flat cache row of every token the oracle writes, and its (b, s)."""
    import oracle
    index = case.index.numpy()
    rows, bs, ss = [], [], []
    for b in range(case.Bkv):
        for s in range(case.Skv):
            slot = oracle.cache_slot(case.mode, b, s, index, case.Skv, case.d0, case.d1)
            if isinstance(slot, tuple):
                rows.append(slot[0] * case.d1 + slot[1])
                bs.append(b)
                ss.append(s)
    return np.array(rows, dtype=np.int64), np.array(bs, dtype=np.int64), np.array(ss, dtype=np.int64)


def check_robust_kv(case, g_ckv, g_k, rel=ROBUST_REL):
    """Codes bit-identical to the oracle's wherever the oracle's float64 value
    lies farther than `rel` (relative; for the RoPE part relative to the
    size of its terms) from a rounding boundary of the cache type: a wrong
    rounding mode or a systematic error of one unit fails here even though it
    stays within the one-ulp / one-code tolerance. Returns the fraction of
    written elements checked."""
    import oracle
    kv, gamma, cos, sin, _ = oracle_kv_inputs(case)
    vy, vr, mr = oracle.kv_values(
        kv, gamma, cos, sin, Dv=case.Dv, eps=f32_arg(case.eps),
        ckv_scale=None if case.ckv_scale is None else case.ckv_scale.numpy(),
        k_scale=None if case.k_scale is None else case.k_scale.numpy(), kc_scale=f32_arg(case.kc_scale))
    rows, bs, ss = kv_token_rows(case)
    checked, total = 0, 0
    for g, v, m, dt, width in ((g_ckv, vy, None, case.ckv_dtype, case.Dv), (g_k, vr, mr, case.k_dtype, case.Dk)):
        gv = np.asarray(g).reshape(-1, width)[rows]
        vt = v[bs, ss]
        margin = rel * (np.abs(vt) if m is None else m[bs, ss])
        want, robust = robust_codes(vt, margin, dt)
        bad = robust & (gv != want)
        assert not bad.any(), "%d codes differ from the oracle away from any rounding boundary (%s), e.g. gpu %s want %s" % (
            int(bad.sum()), dt, gv[bad][:4], want[bad][:4])
        checked += int(robust.sum())
        total += robust.size
    return checked / total if total else 1.0


def oracle_qsa_inputs(case):
    return dict(raw=f64(case.raw), key_length=case.key_length.numpy(),
                rope_cos=f64(case.rope_cos), rope_sin=f64(case.rope_sin),
                k_norm_weight=f64(case.k_norm_weight), past_raw=f64(case.past_raw),
                past_rope=f64(case.past_rope), key_block_size=case.kbs, eps=f32_arg(case.eps))


def run_oracle_qsa(case, block_keys=None, carry=False, rope_layout="interleave_last",
                   past_block_keys=None, values_out=None):
    """past_block_keys: codes [N, Bp, Di] (numpy) for the concat-output form;
    values_out: dict receiving the oracle's pre-rounding keys (see ref_qsa_prepare)."""
    import oracle
    from attention_prologue_kv_gb300.workloads import SENTINEL16
    if block_keys is None:
        block_keys = np.full((case.N, case.Bcap, case.Di), SENTINEL16, dtype=np.uint16)
    nr = npr = None
    if carry:
        nr = np.full((case.N, case.kbs - 1, case.Di), np.nan)
        npr = np.full((case.N, 2 * case.Dr), np.nan) if case.Dr else None
    st = oracle.ref_qsa_prepare(block_keys=block_keys, next_raw=nr, next_rope=npr,
                                rope_layout=rope_layout, past_block_keys=past_block_keys,
                                values_out=values_out,
                                out_dtype="f16" if case.raw.dtype == torch.float16 else "bf16",
                                **oracle_qsa_inputs(case))
    return block_keys, nr, npr, st


QSA_ROBUST_REL = 2.0 ** -17   # float32 error of the block sum and the rotation: at most ~2**-18 of the terms


def check_robust_qsa(g_bk, values, dtype, rel=QSA_ROBUST_REL):
    """Block keys bit-identical to the oracle's wherever its float64 key lies
    farther than `rel` times the magnitude bound of its terms from a rounding
    boundary (values: the oracle's values_out). Returns the fraction checked."""
    checked, total = 0, 0
    for (n, j), (u, b) in values.items():
        want, robust = robust_codes(u, rel * b, dtype)
        got = np.asarray(g_bk)[n, j]
        bad = robust & (got != want)
        assert not bad.any(), "block (%d, %d): %d elements differ away from any rounding boundary" % (
            n, j, int(bad.sum()))
        checked += int(robust.sum())
        total += robust.size
    return checked / total if total else 1.0


# ---------------------------------------------------------------------------
# GPU side (public Python API of the package only)
# ---------------------------------------------------------------------------

def kv_to_device(case, dev="cuda"):
    """The case's kv on the device, keeping a strided-row layout when the case has one."""
    D = case.Dv + case.Dk
    if case.meta.get("row_pad"):
        return case.meta["wide"].to(dev)[:, :D].view(case.Bkv, 1, case.Skv, D)
    return case.kv.to(dev)


def sentinel_cache(shape, dtype, dev="cuda"):
    from attention_prologue_kv_gb300.workloads import TORCH_DTYPES, code_torch_dtype, sentinel
    return torch.full(shape, sentinel(dtype), dtype=code_torch_dtype(dtype), device=dev).view(TORCH_DTYPES[dtype])


GUARD_BYTES = 8192      # guard band before and after every output buffer the kernels write
GUARD_BYTE = 0x5A       # its fill, checked byte for byte after the call


def guarded(shape, dtype, fill, dev="cuda"):
    """An output buffer of `shape` and torch `dtype` filled with `fill`, placed
    between two GUARD_BYTES guard bands inside one allocation (16-byte
    alignment kept). Returns (view, check); check() asserts that no byte of
    either band changed, i.e. that nothing was written outside the buffer."""
    esz = torch.empty(0, dtype=dtype).element_size()
    n = 1
    for d in shape:
        n *= int(d)
    raw = torch.full((GUARD_BYTES * 2 + n * esz,), GUARD_BYTE, dtype=torch.uint8, device=dev)
    view = raw[GUARD_BYTES:GUARD_BYTES + n * esz].view(dtype).view(shape)
    view.fill_(fill)

    def check():
        lo, hi = raw[:GUARD_BYTES], raw[GUARD_BYTES + n * esz:]
        assert bool(torch.all(lo == GUARD_BYTE)) and bool(torch.all(hi == GUARD_BYTE)), \
            "a kernel wrote outside its output buffer (guard band changed)"
    return view, check


def guarded_cache(shape, dtype, dev="cuda"):
    """sentinel_cache between guard bands: (view, check)."""
    from attention_prologue_kv_gb300.workloads import TORCH_DTYPES, code_torch_dtype, sentinel
    v, check = guarded(shape, code_torch_dtype(dtype), sentinel(dtype), dev)
    return v.view(TORCH_DTYPES[dtype]), check


def run_gpu_kv(case, kv=None, ckv=None, k=None, dev="cuda", params_ready=False):
    """Run the CUDA path on a KVCase; returns (ckv codes, k codes, status) as numpy/int."""
    import attention_prologue_kv_gb300 as kvr
    sh_ckv, sh_k = case.cache_shapes()
    checks = []
    if ckv is None:
        ckv, c1 = guarded_cache(sh_ckv, case.ckv_dtype, dev)
        k, c2 = guarded_cache(sh_k, case.k_dtype, dev)
        checks = [c1, c2]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kvr.kv_rmsnorm_rope_cache(
        kv_to_device(case, dev) if kv is None else kv, case.gamma.to(dev), case.cos.to(dev),
        case.sin.to(dev), case.index.to(dev), ckv, k, cache_mode=case.mode, eps=case.eps,
        ckv_scale=None if case.ckv_scale is None else case.ckv_scale.to(dev),
        k_scale=None if case.k_scale is None else case.k_scale.to(dev),
        kc_scale=case.kc_scale, dev_status=status, params_ready=params_ready)
    torch.cuda.synchronize()
    for c in checks:
        c()
    return codes_of(ckv), codes_of(k), int(status.item())


def compare_cache(gpu, ref, dtype, D):
    """Bit-exact on every row the oracle left untouched; on written rows,
    |gpu - ref| <= 2**-7 * |ref| + 1e-6 for 16-bit types, at most one code
    apart on the ordered code line for 8-bit types. Returns (rows written,
    fraction of written elements that are bit-identical)."""
    from attention_prologue_kv_gb300.workloads import sentinel
    from oracle import encoders as enc
    g = gpu.reshape(-1, D)
    r = ref.reshape(-1, D)
    written = ~np.all(r == sentinel(dtype), axis=1)
    untouched_ok = np.array_equal(g[~written], r[~written])
    assert untouched_ok, "bytes outside the indexed rows changed (%d rows)" % int(
        np.sum(~np.all(g[~written] == r[~written], axis=1)))
    gw, rw = g[written], r[written]
    if dtype in ("bf16", "f16"):
        gv, rv = enc.decode(gw, dtype), enc.decode(rw, dtype)
        err = np.abs(gv - rv)
        bad = ~(err <= 2.0**-7 * np.abs(rv) + 1e-6)
        assert not bad.any(), "%d elements out of tolerance, e.g. gpu %s ref %s" % (
            int(bad.sum()), gv[bad][:4], rv[bad][:4])
    else:
        d = np.abs(enc.code_ordinal(gw, dtype) - enc.code_ordinal(rw, dtype))
        assert d.max(initial=0) <= 1, "codes differ by %d" % int(d.max())
    return int(written.sum()), float(np.mean(gw == rw)) if gw.size else 1.0


def run_gpu_qsa(case, carry=False, block_keys=None, dev="cuda", rope_layout="interleave_last",
                past_block_keys=None, params_ready=False, late_key_length=None, key_length_late=False):
    """past_block_keys: codes [N, Bp, Di] (numpy) for the concat-output form.
    late_key_length: the device key_length starts out holding these values
    (int64 tensor shaped like case.key_length), and a kernel launched just
    before the call, which lets the call start at once, writes the case's
    key_length only after a delay (kvr.store_after_delay): the call must use
    the late values."""
    import attention_prologue_kv_gb300 as kvr
    from attention_prologue_kv_gb300.workloads import SENTINEL16
    bk = block_keys
    checks = []
    if bk is None:
        bk, c = guarded((case.N, case.Bcap, case.Di), torch.int16, SENTINEL16, dev)
        bk = bk.view(case.raw.dtype)
        checks.append(c)
    nr = npr = None
    if carry:
        nr, c = guarded((case.N, case.kbs - 1, case.Di), case.raw.dtype, float("nan"), dev)
        checks.append(c)
        if case.Dr:
            npr, c = guarded((case.N, 2 * case.Dr), case.raw.dtype, float("nan"), dev)
            checks.append(c)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    d = lambda t: None if t is None else t.to(dev)
    # every input on the device first: a copy enqueued between the late store
    # and the call would serialise them
    ins = [d(t) for t in (case.raw, case.key_length, case.rope_cos, case.rope_sin, case.k_norm_weight,
                          case.past_raw, case.past_rope)]
    pbk = None if past_block_keys is None else \
        torch.from_numpy(past_block_keys.view(np.int16)).to(dev).view(case.raw.dtype)
    if late_key_length is not None:
        kl = ins[1]
        true_kl = kl.clone()
        kl.copy_(late_key_length.reshape(kl.shape))
        kvr.store_after_delay(kl, true_kl, delay_us=200)
    kvr.qsa_prepare(ins[0], bk, ins[1], ins[2], ins[3], ins[4], ins[5], ins[6], case.kbs, case.eps,
                    next_incomplete_raw_keys=nr, next_incomplete_rope=npr, dev_status=status,
                    rope_layout=rope_layout, past_block_index_keys=pbk, params_ready=params_ready,
                    key_length_late=key_length_late)
    torch.cuda.synchronize()
    for c in checks:
        c()
    return codes_of(bk), f64(nr), f64(npr), int(status.item())


DQ_NEAR_TIE = 2.0 ** -14   # DynamicQuant quotients this close to a half-integer may round either way


def compare_dynamic_quant(g_codes, g_scale, q64, exact=False):
    """DynamicQuant GPU results against the float64 oracle on rows q64.

    Scales: RowMax/127 rounded once to float32 on both sides, so equal.
    Codes: within one code of round-half-even(q*127/RowMax); equal wherever
    that quotient is at least DQ_NEAR_TIE from a half-integer (the kernel's
    reciprocal product is within 2^-15.4 of it); with exact, equal
    everywhere. Returns the fraction of equal codes."""
    from oracle.dynamic_quant import dynamic_quant_quotients, ref_dynamic_quant
    codes, s = ref_dynamic_quant(q64)
    v, _ = dynamic_quant_quotients(q64)
    g = np.asarray(g_codes).reshape(codes.shape)
    assert np.array_equal(np.asarray(g_scale).reshape(-1), s), "scales differ"
    d = np.abs(g.astype(np.int64) - codes.astype(np.int64))
    assert d.max(initial=0) <= 1, "codes differ by %d" % int(d.max())
    if exact:
        assert d.max(initial=0) == 0, "%d codes differ in exact mode" % int((d > 0).sum())
    else:
        far = np.abs(np.abs(v - np.rint(v)) - 0.5) >= DQ_NEAR_TIE
        assert np.array_equal(g[far], codes[far]), "%d codes away from a tie differ" % int(
            (g[far] != codes[far]).sum())
    return float(np.mean(d == 0)) if d.size else 1.0
