"""GPU parity of dynamic_quant against the float64 oracle.

Scales: both sides give RowMax/127 rounded once to float32 (the kernel by
an IEEE division, the oracle by a float64 division that provably rounds to
the same float32), so they must be equal. Codes: within one code of the
oracle's round-half-even(q*127/RowMax) (the tolerance of the int8/FP8
codes), and equal to it wherever that quotient is at least 2^-14 away from
a half-integer (the kernel's reciprocal product is within 2^-15.4 of it).
With exact=True every code must equal the oracle's."""
import numpy as np
import pytest
import torch

import attention_prologue_kv_gb300 as kvr
from attention_prologue_kv_gb300 import workloads as wl
from helpers import compare_dynamic_quant, guarded

pytestmark = pytest.mark.gpu


def check(q_cpu, q_dev=None, exact=False):
    """Returns the fraction of codes equal to the oracle's."""
    q_dev = q_cpu.cuda() if q_dev is None else q_dev
    H = q_cpu.shape[-1]
    out, c1 = guarded(tuple(q_cpu.shape), torch.int8, 99)
    scale, c2 = guarded(tuple(q_cpu.shape[:-1]) + (1,), torch.float32, -1.0)
    kvr.dynamic_quant(q_dev, out, scale, exact=exact)
    torch.cuda.synchronize()
    c1()
    c2()
    return compare_dynamic_quant(out.cpu().numpy(), scale.cpu().numpy(),
                                 q_cpu.reshape(-1, H).to(torch.float64).numpy(), exact)


@pytest.mark.parametrize("exact", [False, True])
def test_decode_workload_full_size(exact):
    q = wl.dynamic_quant_decode()
    assert q.shape == (256, 128, 512)
    assert check(q, exact=exact) > 0.99


@pytest.mark.parametrize("exact", [False, True])
@pytest.mark.parametrize("H", [512, 8, 24, 128, 256, 1024, 1000, 7, 1, 2048])
def test_shapes(H, exact):
    check(wl.dynamic_quant_decode(seed=H, T=5, heads=7, Hckv=H), exact=exact)


@pytest.mark.parametrize("exact", [False, True])
def test_f16_and_strided_rows(exact):
    check(wl.dynamic_quant_decode(seed=3, T=9, heads=5, Hckv=512, dtype="f16"), exact=exact)
    q = wl.dynamic_quant_decode(seed=4, T=9, heads=5, Hckv=512, row_pad=64)
    assert not q.is_contiguous()
    wide = q._base if q._base is not None else q
    check(q.contiguous(), q_dev=wide.cuda()[..., :512], exact=exact)


@pytest.mark.parametrize("exact", [False, True])
def test_zero_rows_and_ties(exact):
    q = wl.dynamic_quant_decode(seed=5, T=4, heads=3, Hckv=64)
    q[1, 2] = 0
    q[2, 0] = torch.tensor([2.5, -3.5, 127.0, 0.5] * 16, dtype=torch.float32).to(q.dtype)
    check(q, exact=exact)


def test_extreme_magnitudes():
    """Rows whose maximum is huge (q*127 would overflow float32 without the
    exact path's rescaling) or tiny (the reciprocal of the scale is not a
    normal float: the exact path throughout)."""
    q = wl.dynamic_quant_decode(seed=6, T=4, heads=4, Hckv=512).float()
    q[0] *= 2.0 ** 120
    q[1] *= 2.0 ** 100
    q[2] *= 2.0 ** -110
    q[3] *= 2.0 ** -125
    q = q.to(torch.bfloat16)
    assert torch.isfinite(q.float()).all()
    for exact in (False, True):
        check(q, exact=exact)


def test_empty():
    q = torch.zeros(0, 4, 512, dtype=torch.bfloat16)
    out = torch.zeros(0, 4, 512, dtype=torch.int8, device="cuda")
    scale = torch.zeros(0, 4, 1, dtype=torch.float32, device="cuda")
    kvr.dynamic_quant(q.cuda(), out, scale)


@pytest.mark.parametrize("exact", [False, True])
def test_ties_and_near_ties_on_power_of_two_scales(exact):
    """Rows with RowMax = 127 * 2**e put q = (k + 1/2) * 2**e exactly halfway
    between codes; their bf16 neighbours lie just off the boundary. The
    oracle rounds ties to even; the default kernel may land on either side of
    an exact tie (one code) but must round the neighbours like the oracle;
    the exact mode must match every code."""
    rows = []
    rng = np.random.default_rng(0)
    for e in (-20, -7, -1, 0, 3, 11):
        m = 127.0 * 2.0 ** e
        k = rng.integers(0, 127, 511)
        ties = (k + 0.5) * 2.0 ** e * rng.choice([-1.0, 1.0], 511)
        t16 = torch.tensor(ties, dtype=torch.float32).to(torch.bfloat16)
        up = (t16.view(torch.int16) + 1).view(torch.bfloat16)
        dn = (t16.view(torch.int16) - 1).view(torch.bfloat16)
        for body in (t16, up, dn):
            rows.append(torch.cat([torch.tensor([m], dtype=torch.bfloat16), body]))
    q = torch.stack(rows).view(len(rows), 1, 512)
    check(q, exact=exact)
    # and scales that are not powers of two, with values crafted near k + 1/2
    q2 = wl.dynamic_quant_decode(seed=9, T=64, heads=4, Hckv=512).float()
    s = q2.abs().amax(-1, keepdim=True) / 127
    near = (torch.round(q2 / s) + 0.5) * s
    check(near.to(torch.bfloat16), exact=exact)
