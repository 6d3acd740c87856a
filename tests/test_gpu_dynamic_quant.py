"""GPU parity of dynamic_quant against the oracle: int8 codes and float32
scales bit-exact (both sides take the same float32 IEEE operations)."""
import numpy as np
import pytest
import torch

import attention_prologue_kv_gb300 as kvr
from attention_prologue_kv_gb300 import workloads as wl
from helpers import guarded
from oracle.dynamic_quant import ref_dynamic_quant

pytestmark = pytest.mark.gpu


def check(q_cpu, q_dev=None):
    q_dev = q_cpu.cuda() if q_dev is None else q_dev
    H = q_cpu.shape[-1]
    out, c1 = guarded(tuple(q_cpu.shape), torch.int8, 99)
    scale, c2 = guarded(tuple(q_cpu.shape[:-1]) + (1,), torch.float32, -1.0)
    kvr.dynamic_quant(q_dev, out, scale)
    torch.cuda.synchronize()
    c1()
    c2()
    codes, s = ref_dynamic_quant(q_cpu.reshape(-1, H).to(torch.float64).numpy())
    assert np.array_equal(out.cpu().reshape(-1, H).numpy(), codes)
    assert np.array_equal(scale.cpu().reshape(-1).numpy(), s)


def test_decode_workload_full_size():
    q = wl.dynamic_quant_decode()
    assert q.shape == (256, 128, 512)
    check(q)


@pytest.mark.parametrize("H", [512, 8, 24, 128, 256, 1024, 1000, 7, 1, 2048])
def test_shapes(H):
    check(wl.dynamic_quant_decode(seed=H, T=5, heads=7, Hckv=H))


def test_f16_and_strided_rows():
    check(wl.dynamic_quant_decode(seed=3, T=9, heads=5, Hckv=512, dtype="f16"))
    q = wl.dynamic_quant_decode(seed=4, T=9, heads=5, Hckv=512, row_pad=64)
    assert not q.is_contiguous()
    wide = q._base if q._base is not None else q
    check(q.contiguous(), q_dev=wide.cuda()[..., :512])


def test_zero_rows_and_ties():
    q = wl.dynamic_quant_decode(seed=5, T=4, heads=3, Hckv=64)
    q[1, 2] = 0
    q[2, 0] = torch.tensor([2.5, -3.5, 127.0, 0.5] * 16, dtype=torch.float32).to(q.dtype)
    check(q)


def test_empty():
    q = torch.zeros(0, 4, 512, dtype=torch.bfloat16)
    out = torch.zeros(0, 4, 512, dtype=torch.int8, device="cuda")
    scale = torch.zeros(0, 4, 1, dtype=torch.float32, device="cuda")
    kvr.dynamic_quant(q.cuda(), out, scale)


def test_ties_and_near_ties_on_power_of_two_scales():
    """Rows with RowMax = 127 * 2**e have scale exactly 2**e, so q = (k + 1/2) * 2**e
    lands exactly halfway between codes; their bf16 neighbours lie just off the
    boundary. Every element must round exactly like the oracle's float32 division."""
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
    check(q)
    # and scales that are not powers of two, with values crafted near k + 1/2
    q2 = wl.dynamic_quant_decode(seed=9, T=64, heads=4, Hckv=512).float()
    s = q2.abs().amax(-1, keepdim=True) / 127
    near = (torch.round(q2 / s) + 0.5) * s
    check(near.to(torch.bfloat16))
