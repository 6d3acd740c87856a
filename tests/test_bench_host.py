"""Host logic of the benchmark without a GPU: the algorithmic byte model and
the replica timing reduction over two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_algorithmic_bytes_match_the_hand_count():
    # decode: 251 active tokens x (1152 kv + 256 cos/sin + 8 index + 1024 ckv + 128 k) + 5 x 8 + 1024 gamma
    assert bench.kv_algorithmic_bytes(251, 5) == 251 * 2568 + 40 + 1024 == 645632
    # prefill: 32768 tokens, no skips
    assert bench.kv_algorithmic_bytes(32768, 0) == 84149248
    # FP8 ckv: 512-byte rows, plus the 2048-byte per-channel scale
    assert bench.kv_algorithmic_bytes(4096, 0, ckv_bytes=1, scale_bytes=2048) == 4096 * 2056 + 1024 + 2048
    # QSA: 32 sequences x 32 blocks x (64 rows x 256 B + 256 B cos/sin + 256 B key) + 32 x 8 + 256
    assert bench.qsa_algorithmic_bytes(1024, 32, 64, 128, 64) == 17302016


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, tok = bench.reduce_timing(10.0 + 5 * rank, 1000 * (rank + 1))
        bench.barrier()
        out[rank] = (ms, tok)
    finally:
        dist.destroy_process_group()


def test_replica_timing_reduction_two_ranks():
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, start_method="spawn")
    assert out[0] == out[1] == (15.0, 3000.0)


def test_reduce_timing_without_process_group_is_identity():
    assert bench.reduce_timing(3.5, 42) == (3.5, 42.0)


def test_default_arguments_obey_the_contract():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.impl == "ours"
    assert bench.parse_args(["--warmup", "0"]).warmup == 3


def test_kernel_source_hash_ignores_comments_not_code():
    """The profiled-traffic guard keys on code: comments and layout do not
    change it, any code or string-literal change does."""
    import bench
    a = 'x = 1; // note\n/* block\n comment */ asm("mov // not a comment");'
    b = 'x = 1;\n\n   asm("mov // not a comment");   // other note'
    assert bench._code_tokens(a) == bench._code_tokens(b)
    assert bench._code_tokens(a) != bench._code_tokens(a.replace("x = 1", "x = 2"))
    assert bench._code_tokens(a) != bench._code_tokens(a.replace("mov //", "mov2 //"))


def test_cpu_baseline_on_several_processes():
    """The oracle baseline in spawned processes (one per host core in the
    benchmark; two here): every process reports, the aggregate counts all of
    them, and each process's rate is of the order of the single-process rate."""
    from attention_prologue_kv_gb300 import workloads as wl
    case = wl.make_kv_case("b", 2, 256, mode="PA_BSND", d0=16, d1=128, seed=1003, slots="table", pos="seq")
    one = bench.cpu_oracle_baseline(0.5, case)
    res = bench.cpu_oracle_all_cores(0.5, case, n=2)
    assert res is not None
    tps, procs, seqs, secs = res
    assert procs == 2 and seqs >= 2 and secs >= 0.5
    assert 0.1 * one[0] < tps / procs < 10 * one[0]


def test_algorithmic_bytes_of_the_workloads():
    """The bytes each workload must move, worked out by hand from its sizes:
    decode 251 active rows x (1152 kv + 256 cos/sin + 8 index + 1024 + 128
    cache) + 5 skipped index entries + 1 KB gamma; prefill 32768 rows; the FP8
    workload with 512-byte ckv rows and a 2 KB scale; QSA 1024 blocks of 64
    rows x 256 B + first-token cos/sin 256 B + key 256 B, 32 key_length
    entries, 256 B weight; DynamicQuant 32768 rows of 1024 + 512 + 4 B."""
    assert bench.kv_algorithmic_bytes(251, 5) == 251 * 2568 + 5 * 8 + 1024 == 645632
    assert bench.kv_algorithmic_bytes(32768, 0) == 84149248
    assert bench.kv_algorithmic_bytes(4096, 0, ckv_bytes=1, scale_bytes=2048) == 4096 * 2056 + 1024 + 2048
    assert bench.qsa_algorithmic_bytes(1024, 32, 64, 128, 64) == 1024 * (16384 + 256 + 256) + 256 + 256 == 17302016
    assert bench.dq_algorithmic_bytes(32768, 512) == 32768 * 1540 == 50462720


def test_prefill_rotation_writes_disjoint_rows():
    """The benchmark's rotated prefill batches write disjoint cache blocks,
    each batch 32768 distinct slots, contiguous within each 128-slot block:
    no call rewrites a row another call of the rotation wrote."""
    import torch
    from attention_prologue_kv_gb300 import workloads as wl
    cases = bench.prefill_sets(bench.ROTATION)
    blocks = [set((c.index // 128).tolist()) for c in cases]
    assert all(len(b) == 256 for b in blocks)
    assert len(set.union(*blocks)) == 256 * len(cases)
    for c in cases:
        idx = c.index.view(8, 4096)
        assert len(set(c.index.tolist())) == 32768
        assert torch.all((idx[:, 1:] - idx[:, :-1])[:, torch.arange(4095) % 128 != 127] == 1)
