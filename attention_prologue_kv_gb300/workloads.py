"""Seeded synthetic inputs for the KV prologue and the QSA block-key prepare.

This module is the one piece that both the CUDA path's tests/benchmark and
the oracle consume. It only draws random numbers and builds RoPE tables and
slot indices; it holds none of the normalisation, rotation, quantisation or
placement arithmetic. All tensors are created on the CPU from a
torch.Generator with a fixed seed; callers copy them to the device.

RoPE tables: angle(pos, j) = pos * base**(-2*(j mod h)/W) for a table of
width W = 2h, so lanes j and j + h share one angle (cos^2 + sin^2 = 1 per
output pair), computed in float64, stored in the input dtype.
"""
import math
from dataclasses import dataclass, field

import torch

SENTINEL16 = 0x7FBF   # a bfloat16 NaN pattern: no finite result encodes to it
SENTINEL8 = 0x7F      # NaN for both FP8 formats, 127 for int8

TORCH_DTYPES = {
    "bf16": torch.bfloat16,
    "f16": torch.float16,
    "int8": torch.int8,
    "fp8_e4m3fn": torch.float8_e4m3fn,
    "fp8_e5m2": torch.float8_e5m2,
}


def code_torch_dtype(dtype):
    """Integer container torch dtype holding the bit patterns of `dtype`."""
    return torch.int16 if dtype in ("bf16", "f16") else torch.uint8


def sentinel(dtype):
    return SENTINEL16 if dtype in ("bf16", "f16") else SENTINEL8


def rope_tables(pos, width, base=10000.0, dtype=torch.bfloat16):
    """cos/sin tables [*pos.shape, width] for integer positions `pos`."""
    h = width // 2
    j = torch.arange(width, dtype=torch.float64) % h
    inv = base ** (-2.0 * j / width)
    ang = pos.to(torch.float64).unsqueeze(-1) * inv
    return torch.cos(ang).to(dtype), torch.sin(ang).to(dtype)


@dataclass
class KVCase:
    """One synthetic call of the KV prologue (all tensors on the CPU)."""
    name: str
    Bkv: int
    Skv: int
    Dv: int
    Dk: int
    mode: str                 # "Norm" | "PA_BSND" | "PA_BLK_BSND"
    d0: int                   # Bcache or BlockNum
    d1: int                   # Scache or BlockSize
    ckv_dtype: str
    k_dtype: str
    eps: float
    kv: torch.Tensor          # [Bkv, 1, Skv, D] (or a column slice of a wider row)
    gamma: torch.Tensor       # [Dv]
    cos: torch.Tensor         # [Bkv, 1, Skv, Dk]
    sin: torch.Tensor
    index: torch.Tensor       # int64, layout per mode
    ckv_scale: torch.Tensor = None   # float32 [Dv] or [1] for an 8-bit ckv cache
    k_scale: torch.Tensor = None     # float32 [Dk] or [1] for an 8-bit k cache
    kc_scale: float = 1.0
    meta: dict = field(default_factory=dict)

    @property
    def T(self):
        return self.Bkv * self.Skv

    def cache_shapes(self):
        return (self.d0, self.d1, 1, self.Dv), (self.d0, self.d1, 1, self.Dk)

    def active_tokens(self):
        """Tokens whose index entry is not -1 (for byte counting)."""
        if self.mode == "PA_BLK_BSND":
            nb = -(-self.Skv // self.d1)
            ent = self.index.view(self.Bkv, nb)
            s = torch.arange(self.Skv)
            return int((ent[:, s // self.d1] != -1).sum())
        return int((self.index != -1).sum())


def make_kv_case(name, Bkv, Skv, Dv=512, Dk=64, mode="PA_BSND", d0=None, d1=128,
                 ckv_dtype="bf16", k_dtype="bf16", seed=0, kv_std=1.0,
                 skip=0, slots="random", pos="random", pos_max=32768,
                 scale_len=None, kc_scale=1.0, eps=1e-6, in_dtype="bf16",
                 row_pad=0, k_scale_len=None):
    """Build a KVCase.

    skip      number of index entries set to -1 (chosen at random)
    slots     "random": distinct random slots over the whole cache;
              "table": a random per-sequence block table, contiguous within a block
    pos       "random": one random position per token in [0, pos_max);
              "start": a random start in [0, pos_max) per sequence, + s;
              "seq": position s
    row_pad   extra elements after each kv row (kv becomes a [Bkv, 1, Skv, D]
              view of a wider [T, D + row_pad] buffer: strided rows)
    """
    g = torch.Generator().manual_seed(seed)
    dt = TORCH_DTYPES[in_dtype]
    D = Dv + Dk
    T = Bkv * Skv
    wide = torch.randn(T, D + row_pad, generator=g, dtype=torch.float32) * kv_std
    wide = wide.to(dt)
    kv = wide[:, :D].view(Bkv, 1, Skv, D)   # strided rows when row_pad > 0
    gamma = (torch.rand(Dv, generator=g, dtype=torch.float32) + 0.5).to(dt)

    if pos == "random":
        p = torch.randint(0, pos_max, (Bkv, Skv), generator=g)
    elif pos == "start":
        p = torch.randint(0, pos_max, (Bkv, 1), generator=g) + torch.arange(Skv)
    else:
        p = torch.arange(Skv).expand(Bkv, Skv)
    cos, sin = rope_tables(p, Dk, dtype=dt)
    cos = cos.view(Bkv, 1, Skv, Dk)
    sin = sin.view(Bkv, 1, Skv, Dk)

    if mode == "Norm":
        if d0 is None:
            d0 = Bkv
        index = torch.stack([torch.randperm(d1, generator=g)[:Skv] for _ in range(Bkv)])
        flat = index.view(-1)
    elif mode == "PA_BSND":
        if slots == "table":
            nb = -(-Skv // d1)
            table = torch.randperm(d0, generator=g)[:Bkv * nb].view(Bkv, nb)
            s = torch.arange(Skv)
            index = (table[:, s // d1] * d1 + s % d1).reshape(-1)
        else:
            index = torch.randperm(d0 * d1, generator=g)[:T]
        flat = index
    elif mode == "PA_BLK_BSND":
        nb = -(-Skv // d1)
        index = torch.randperm(d0, generator=g)[:Bkv * nb] * d1
        flat = index
    else:
        raise ValueError(mode)
    if skip:
        flat[torch.randperm(flat.numel(), generator=g)[:skip]] = -1
    index = index.contiguous().to(torch.int64)

    ckv_scale = k_scale = None
    if ckv_dtype not in ("bf16", "f16"):
        n = scale_len if scale_len is not None else Dv
        ckv_scale = torch.rand(n, generator=g, dtype=torch.float32) * 1.5 + 0.5
    if k_dtype not in ("bf16", "f16"):
        n = k_scale_len if k_scale_len is not None else Dk
        k_scale = torch.rand(n, generator=g, dtype=torch.float32) * 1.5 + 0.5

    return KVCase(name=name, Bkv=Bkv, Skv=Skv, Dv=Dv, Dk=Dk, mode=mode, d0=d0, d1=d1,
                  ckv_dtype=ckv_dtype, k_dtype=k_dtype, eps=eps, kv=kv, gamma=gamma,
                  cos=cos, sin=sin, index=index, ckv_scale=ckv_scale, k_scale=k_scale,
                  kc_scale=kc_scale, meta=dict(seed=seed, kv_std=kv_std, pos=pos,
                                               slots=slots, skip=skip, in_dtype=in_dtype,
                                               row_pad=row_pad, wide=wide))


# The five synthetic workloads (seed = 1000 + workload number).
def tiny_norm(seed=1001):
    """Bkv=2, Skv=16, Norm cache [2, 32, 1, 512|64], ~10% of indices -1."""
    return make_kv_case("tiny_norm", 2, 16, mode="Norm", d0=2, d1=32, seed=seed,
                        skip=3, pos="start", pos_max=1000)


def decode_paged(seed=1002):
    """Bkv=256, Skv=1, PA_BSND BlockSize=128 BlockNum=4096, 2% of indices -1."""
    return make_kv_case("decode_paged", 256, 1, mode="PA_BSND", d0=4096, d1=128,
                        seed=seed, skip=round(0.02 * 256), pos="random", pos_max=32768)


def prefill_paged(seed=1003):
    """Bkv=8, Skv=4096, kv std 2, PA_BSND BlockSize=128 BlockNum=2048, block table."""
    return make_kv_case("prefill_paged", 8, 4096, mode="PA_BSND", d0=2048, d1=128,
                        seed=seed, kv_std=2.0, slots="table", pos="seq")


def quant_fp8(seed=1004):
    """Bkv=64, Skv=64, FP8-E4M3FN ckv cache with per-channel scale, bf16 k cache."""
    return make_kv_case("quant_fp8", 64, 64, mode="PA_BSND", d0=1024, d1=128,
                        ckv_dtype="fp8_e4m3fn", seed=seed, pos="random", pos_max=32768)


@dataclass
class QSACase:
    """One synthetic call of the QSA block-key prepare (CPU tensors)."""
    name: str
    N: int
    L: int
    Di: int
    Dr: int
    kbs: int
    eps: float
    Bcap: int
    raw: torch.Tensor            # [N, L, Di]
    key_length: torch.Tensor     # int64 [N] or [1]
    rope_cos: torch.Tensor       # [N, L, Dr] or None
    rope_sin: torch.Tensor
    k_norm_weight: torch.Tensor  # [Di] or None
    past_raw: torch.Tensor       # [N, kbs-1, Di]
    past_rope: torch.Tensor      # [N, 2*Dr] or None
    meta: dict = field(default_factory=dict)

    def completed_blocks(self):
        K = self.key_length.expand(self.N) if self.key_length.numel() == 1 else self.key_length
        P = K - self.L
        return int(((K // self.kbs) - (P // self.kbs)).clamp(min=0).sum())


def make_qsa_case(name, N, L, Di=128, Dr=64, kbs=64, seed=0, past_max=8192,
                  past=None, rope=True, norm=True, eps=1e-6, Bcap=None,
                  shared_length=False, in_dtype="bf16"):
    """Build a QSACase. Past lengths are drawn from [0, past_max) unless
    `past` (a list) is given; carry rows at or beyond the incomplete fill f
    are NaN (they must never be read), as is past_rope when f = 0."""
    g = torch.Generator().manual_seed(seed)
    dt = TORCH_DTYPES[in_dtype]
    raw = torch.randn(N, L, Di, generator=g, dtype=torch.float32).to(dt)
    w = (torch.rand(Di, generator=g, dtype=torch.float32) + 0.5).to(dt) if norm else None
    if past is None:
        if shared_length:
            P = torch.randint(0, past_max, (1,), generator=g).expand(N).clone()
        else:
            P = torch.randint(0, past_max, (N,), generator=g)
    else:
        P = torch.tensor(past, dtype=torch.int64)
    P = P.to(torch.int64)
    f = P % kbs
    key_length = (P + L).to(torch.int64)
    if shared_length:
        key_length = key_length[:1].clone()
    past_raw = torch.randn(N, kbs - 1, Di, generator=g, dtype=torch.float32)
    rows = torch.arange(kbs - 1).unsqueeze(0)
    past_raw[(rows >= f.unsqueeze(1))] = float("nan")
    past_raw = past_raw.to(dt)
    rope_cos = rope_sin = past_rope = None
    if rope:
        pos = P.unsqueeze(1) + torch.arange(L)
        rope_cos, rope_sin = rope_tables(pos, Dr, dtype=dt)
        pc, ps = rope_tables(P - f, Dr, dtype=dt)
        past_rope = torch.cat([pc, ps], dim=-1)
        past_rope[f == 0] = float("nan")
    if Bcap is None:
        Bcap = int((P.max() + L) // kbs) + 1
    return QSACase(name=name, N=N, L=L, Di=Di, Dr=Dr if rope else 0, kbs=kbs, eps=eps,
                   Bcap=Bcap, raw=raw, key_length=key_length, rope_cos=rope_cos,
                   rope_sin=rope_sin, k_norm_weight=w, past_raw=past_raw,
                   past_rope=past_rope, meta=dict(seed=seed, past=P.tolist()))


def qsa_prepare_workload(seed=1005):
    """N=32, L=2048, Di=128, Dr=64, kbs=64, past lengths in [0, 8192), Bcap=160."""
    return make_qsa_case("qsa_prepare", 32, 2048, Di=128, Dr=64, kbs=64, seed=seed,
                         past_max=8192, Bcap=160)


def dynamic_quant_decode(seed=1006, T=256, heads=128, Hckv=512, dtype="bf16", row_pad=0):
    """q^N of one decode step: T tokens x `heads` heads x Hckv, ~N(0, 1), as
    [T, heads, Hckv] (a column slice of wider rows when row_pad > 0)."""
    g = torch.Generator().manual_seed(seed)
    wide = torch.randn(T, heads, Hckv + row_pad, generator=g, dtype=torch.float32).to(TORCH_DTYPES[dtype])
    return wide[..., :Hckv]


KV_WORKLOADS = {
    "tiny_norm": tiny_norm,
    "decode_paged": decode_paged,
    "prefill_paged": prefill_paged,
    "quant_fp8": quant_fp8,
}


def prefill_paged_sets(n_sets, seed=1003):
    """`n_sets` prefill batches shaped like prefill_paged, each from its own
    seed, whose block tables use disjoint cache blocks (n_sets * 256 of the
    2048 blocks, from one random permutation), so that no two batches of a
    rotation write the same cache rows."""
    cases = [prefill_paged(seed=seed + 7919 * i) for i in range(n_sets)]
    c0 = cases[0]
    nb = -(-c0.Skv // c0.d1)
    if n_sets * c0.Bkv * nb > c0.d0:
        raise ValueError("too many sets for disjoint block tables")
    perm = torch.randperm(c0.d0, generator=torch.Generator().manual_seed(seed + 1))
    s = torch.arange(c0.Skv)
    for i, c in enumerate(cases):
        table = perm[i * c.Bkv * nb:(i + 1) * c.Bkv * nb].view(c.Bkv, nb)
        c.index = (table[:, s // c.d1] * c.d1 + s % c.d1).reshape(-1).contiguous().to(torch.int64)
    return cases


def decode_paged_sets(n_sets, seed=1002, Bkv=256, Dv=512, Dk=64, block_num=4096, block_size=128,
                      n_skip=5, pos_max=32768):
    """`n_sets` independent decode batches shaped like decode_paged, stacked:
    kv [n, Bkv, 1, 1, Dv+Dk], cos/sin [n, Bkv, 1, 1, Dk], index [n, Bkv] and
    one gamma [Dv]. All slots are distinct (within and across sets); n_skip
    entries per set are -1. Used to rotate a benchmark's inputs through more
    memory than L2 holds."""
    g = torch.Generator().manual_seed(seed)
    D = Dv + Dk
    kv = (torch.randn(n_sets, Bkv, 1, 1, D, generator=g, dtype=torch.float32)).to(torch.bfloat16)
    gamma = (torch.rand(Dv, generator=g, dtype=torch.float32) + 0.5).to(torch.bfloat16)
    pos = torch.randint(0, pos_max, (n_sets, Bkv), generator=g)
    cos, sin = rope_tables(pos, Dk)
    slots = torch.randperm(block_num * block_size, generator=g)[:n_sets * Bkv].view(n_sets, Bkv).clone()
    if n_skip:
        drop = torch.rand(n_sets, Bkv, generator=g).argsort(dim=1)[:, :n_skip]
        slots.scatter_(1, drop, -1)
    return dict(kv=kv, gamma=gamma, cos=cos.view(n_sets, Bkv, 1, 1, Dk),
                sin=sin.view(n_sets, Bkv, 1, 1, Dk), index=slots.to(torch.int64),
                Dv=Dv, Dk=Dk, d0=block_num, d1=block_size)
