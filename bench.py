#!/usr/bin/env python3
"""Benchmark of the fused KV prologue (RMSNorm + interleaved RoPE + paged
cache scatter) on the prefill workload, plus the other workloads as extras.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one kv_rmsnorm_rope_cache call on one prefill batch: Bkv = 8
sequences x Skv = 4096 tokens (32768 token rows), D = 512 + 64 bf16, kv
~N(0, std 2), positions 0..4095, PA_BSND caches BlockSize 128 x BlockNum
2048 written through a random per-sequence block table. Steps rotate over 4
independent input sets (186 MB > L2) whose block tables are disjoint, so
every step reads its inputs from HBM and writes rows no other step of the
rotation writes. The K timed steps run as CUDA-graph replays of back-to-back
calls (graphs of up to 256 calls cycling through the rotation, plus a
remainder graph; each graph is replayed once, untimed, before the timed
region), timed with CUDA events on the capture stream. With N > 1 (torchrun) each rank runs an independent
replica on its own GPU; the job value sums tokens over ranks and divides by
the slowest rank's time (weak scaling, no data-path collective).

Printed on rank 0: one JSON line with the metric, the roofline of the kernel,
the CPU oracle baseline (one process, and one spawned process per host core
under "all_cores"), the end-to-end figure (host buffers, host<->device
copies inside the timed region), clocks sampled during the timed region, and
the other workloads (decode, FP8 quantised, QSA prepare, DynamicQuant) under
"extras" as microseconds per call and fractions of the measured HBM peak.
"""
import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "tokens/s and achieved HBM GB/s (% of GB300 peak) for fused norm+RoPE+cache write"
UNIT = "tokens/s"
ROTATION = 4             # input sets rotated through by the prefill steps
GRAPH_CALLS = 256        # calls per captured CUDA graph (cycling through the rotation)
DEFAULT_STEPS = 2048     # 512 rotations, ~30 ms of GPU time
DEFAULT_WARMUP = 16
WORKLOAD = ("prefill_paged: Bkv=8 Skv=4096 (32768 tokens) N=1 D=576 (Dv=512 rmsnorm, Dk=64 interleaved RoPE) "
            "bf16, kv ~N(0,std 2), gamma ~U(0.5,1.5), positions 0..4095, PA_BSND bf16 caches BlockSize=128 "
            "BlockNum=2048, slots from a random per-sequence block table (the rotated batches use disjoint blocks)")
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "kv_bulk_kernel__prefill_paged.md")
KERNEL_SOURCES = [os.path.join(ROOT, "attention_prologue_kv_gb300", "csrc", f)
                  for f in ("kv_bulk.cu", "kv_common.cuh", "kvr_internal.cuh")]


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=DEFAULT_STEPS)
    ap.add_argument("--warmup", type=int, default=DEFAULT_WARMUP)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU work budget of the oracle baseline leg")
    ap.add_argument("--no-extras", action="store_true", help="skip the other workloads")
    ap.add_argument("--extras-only", action="store_true", help="time only the other workloads")
    ap.add_argument("--only", choices=["prefill_paged", "quant_fp8", "tiny_norm", "qsa_prepare",
                                       "qsa_prepare_params_ready", "decode_paged", "dynamic_quant_decode",
                                       "dynamic_quant_decode_exact"],
                    help="run W + K launches of one workload and print their timing (for profilers)")
    ap.add_argument("--profile-range", action="store_true",
                    help="with --only: launch the K steps back to back inside one cudaProfilerStart/Stop range "
                         "(no per-launch timing), for a profiler's range replay")
    ap.add_argument("--profile-graph", action="store_true",
                    help="with --profile-range: capture the K steps as one CUDA graph (replayed once untimed "
                         "first) and replay it inside the range, as the benchmark runs them; for an "
                         "application-range replay")
    a = ap.parse_args(argv)
    a.warmup = max(a.warmup, 3)
    a.steps = max(a.steps, 1)
    return a


# ---------------------------------------------------------------------------
# Algorithmic bytes (what the method must move; untouched cache slots and
# -1 rows' inputs are not counted)
# ---------------------------------------------------------------------------

def kv_algorithmic_bytes(n_active, n_skipped, Dv=512, Dk=64, in_bytes=2, ckv_bytes=2, k_bytes=2,
                         scale_bytes=0):
    per_active = (Dv + Dk) * in_bytes + 2 * Dk * in_bytes + 8 + Dv * ckv_bytes + Dk * k_bytes
    return n_active * per_active + n_skipped * 8 + Dv * in_bytes + scale_bytes


def dq_algorithmic_bytes(rows, H, in_bytes=2):
    """DynamicQuant: read the row, write its int8 codes and one float32 scale."""
    return rows * (H * in_bytes + H + 4)


def qsa_algorithmic_bytes(n_blocks, n_seq, kbs, Di, Dr, in_bytes=2):
    per_block = kbs * Di * in_bytes + 2 * Dr * in_bytes + Di * in_bytes
    return n_blocks * per_block + n_seq * 8 + Di * in_bytes


# ---------------------------------------------------------------------------
# Multi-rank plumbing (replicas: only the timing result is exchanged)
# ---------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_timing(elapsed_ms, tokens, device=None):
    """Max of the elapsed time and sum of the tokens over all ranks (identity
    when no process group is initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(elapsed_ms), float(tokens)
    t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
    n = torch.tensor([float(tokens)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), float(n.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# Clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id):
        self.cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                    "-lms", "50", "-i", str(gpu_id)]
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None
        time.sleep(0.3)

    def stop(self, t0, t1):
        if self.p is None:
            return None
        time.sleep(0.15)
        self.p.terminate()
        try:
            out = self.p.communicate(timeout=10)[0]
        except subprocess.TimeoutExpired:
            self.p.kill()
            out = self.p.communicate()[0]
        rows = []
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) != 8:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[1]), float(f[2]), f[4:8]))
            except ValueError:
                continue
        if not rows:
            return None
        inside = [r for r in rows if t0 - 0.06 <= r[0] <= t1 + 0.06]
        window = "timed region"
        if not inside:
            inside = rows
            window = "whole run (timed region shorter than the sampling interval)"
        reasons = sorted({self.REASONS[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


def gpu_smi_id(dev):
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return dev


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def _code_tokens(text):
    """C/C++/CUDA source with comments removed and whitespace runs collapsed
    (string and character literals kept verbatim): what decides the code."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash():
    """Hash of the profiled kernel's sources, blind to comments and layout."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(f, encoding="utf-8") as fh:
            h.update(_code_tokens(fh.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the kernel source as it is now (else None)."""
    try:
        lines = open(PROFILE_SUMMARY).read().splitlines()
    except OSError:
        return None, None
    kv = {}
    for line in lines:
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            kv[k.strip()] = v.strip().strip("`")
    if kv.get("kernel_source_sha256") != kernel_source_hash():
        return None, "stale"
    try:
        return float(kv["traffic_bytes_per_launch"]), "ok"
    except (KeyError, ValueError):
        return None, None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


def l2_flush(buf):
    buf.add_(1)


def time_each(fn, n, flush, stream):
    """Median/min of n single-launch durations (CUDA events on `stream`), L2 flushed before each."""
    import torch
    ts = []
    for _ in range(n):
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts), min(ts)


def _oracle_seqs(case, n):
    """The first n sequences of a PA_BSND KV case as the oracle's float64 /
    int64 arrays, one tuple (kv [1, Skv, D], cos, sin [1, Skv, Dk], index [Skv])
    per sequence, and gamma."""
    D, Dk = case.Dv + case.Dk, case.Dk
    kv = case.kv.double().reshape(case.Bkv, case.Skv, D).numpy()
    cos = case.cos.double().reshape(case.Bkv, case.Skv, Dk).numpy()
    sin = case.sin.double().reshape(case.Bkv, case.Skv, Dk).numpy()
    idx = case.index.numpy().reshape(case.Bkv, case.Skv)
    seqs = [(kv[b:b + 1], cos[b:b + 1], sin[b:b + 1], idx[b]) for b in range(min(n, case.Bkv))]
    return seqs, case.gamma.double().numpy()


def _oracle_loop(budget_s, seqs, gamma, d0, d1, Dv):
    """The oracle as it stands on whole sequences (cycled) for about budget_s
    seconds: (tokens/s, sequences, seconds)."""
    import numpy as np

    import oracle
    Dk = seqs[0][1].shape[-1]
    ckv = np.full((d0, d1, Dv), 0x7FBF, dtype=np.uint16)
    kc = np.full((d0, d1, Dk), 0x7FBF, dtype=np.uint16)
    n_tok, n_seq = 0, 0
    t0 = time.perf_counter()
    while True:
        kv, cos, sin, idx = seqs[n_seq % len(seqs)]
        oracle.ref_kv_rmsnorm_rope_cache(kv, gamma, cos, sin, idx, ckv, kc, Dv=Dv, mode="PA_BSND", eps=1e-6)
        n_tok += kv.shape[1]
        n_seq += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return n_tok / el, n_seq, el


def cpu_oracle_baseline(budget_s, case):
    """The oracle as it stands, on whole sequences of the workload, for about
    budget_s seconds of single-process CPU time: (tokens/s, sequences, s)."""
    seqs, gamma = _oracle_seqs(case, 2)
    return _oracle_loop(budget_s, seqs, gamma, case.d0, case.d1, case.Dv)


def _oracle_process(budget_s, inputs, barrier, out):
    """One process of the all-cores oracle run, timed after every process is
    ready (so that the timed windows overlap)."""
    barrier.wait(timeout=600)
    out.put(_oracle_loop(budget_s, *inputs))


def cpu_oracle_all_cores(budget_s, case, n=None):
    """The same oracle in one process per host core (n processes if given;
    spawned, so no process inherits a CUDA context; each gets one sequence of
    the workload and its own caches), started together: aggregate
    (tokens/s, processes, sequences, seconds)."""
    import multiprocessing as mp
    n = n or os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    barrier, out = ctx.Barrier(n), ctx.Queue()
    seqs, gamma = _oracle_seqs(case, case.Bkv)
    procs = []
    for i in range(n):
        procs.append(ctx.Process(target=_oracle_process,
                                 args=(budget_s, ([seqs[i % len(seqs)]], gamma, case.d0, case.d1, case.Dv),
                                       barrier, out)))
    for p in procs:
        p.start()
    res, deadline = [], time.time() + 600
    while len(res) < n and time.time() < deadline:
        try:
            res.append(out.get(timeout=1.0))
        except Exception:   # queue.Empty: check that no process has failed
            if any(p.exitcode not in (None, 0) for p in procs):
                break
    for p in procs:
        p.join(timeout=5)
        if p.is_alive():
            p.terminate()
    if len(res) < n:
        return None
    return sum(r[0] for r in res), n, sum(r[1] for r in res), max(r[2] for r in res)


def prefill_sets(n, rank=0):
    """n independent prefill batches (CPU tensors) writing disjoint cache
    blocks; the benchmark uses the first one's gamma for all of them (one
    model weight)."""
    from attention_prologue_kv_gb300 import workloads as wl
    return wl.prefill_paged_sets(n, seed=1003 + 100003 * rank)


def run_ours(args):
    import torch
    import torch.distributed as dist

    import attention_prologue_kv_gb300 as kvr

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    from attention_prologue_kv_gb300.build import build
    if rank == 0 or world == 1:
        build()
    barrier()

    # ---- inputs: ROTATION prefill batches resident in HBM ----
    R = ROTATION
    cases = prefill_sets(R, rank)
    c0 = cases[0]
    kv = [c.kv.to(dev) for c in cases]
    cos = [c.cos.to(dev) for c in cases]
    sin = [c.sin.to(dev) for c in cases]
    index = [c.index.to(dev) for c in cases]
    gamma = c0.gamma.to(dev)
    d0, d1 = c0.d0, c0.d1
    ckv = torch.full((d0, d1, 1, c0.Dv), 0x7FBF, dtype=torch.int16, device=dev).view(torch.bfloat16)
    kc = torch.full((d0, d1, 1, c0.Dk), 0x7FBF, dtype=torch.int16, device=dev).view(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    T = c0.T
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    calls = [kvr.prepare_kv_rmsnorm_rope_cache(kv[i], gamma, cos[i], sin[i], index[i], ckv, kc,
                                               cache_mode="PA_BSND", eps=1e-6, dev_status=status)
             for i in range(R)]

    # ---- warm-up: W eager steps ----
    for w in range(args.warmup):
        calls[w % R]()
    torch.cuda.synchronize()

    # ---- graphs of GRAPH_CALLS calls (a multiple of R), plus the remainder;
    # each replayed once untimed. Calls overlap (programmatic dependent
    # launch) only inside a graph, so graphs are long. ----
    K = args.steps
    G = min(GRAPH_CALLS, K) // R * R or K
    full, rem = divmod(K, G)
    graphs = []
    for n in ([G] if full else []) + ([rem] if rem else []):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                calls[i % R]()
        graphs.append(g)
    for g in graphs:
        g.replay()           # graph upload and first-launch costs stay out of the timed region
    torch.cuda.synchronize()
    g_full = graphs[0] if full else None
    g_rem = graphs[-1] if rem else None
    stream = torch.cuda.current_stream()

    sampler = ClockSampler(gpu_smi_id(local)) if rank == 0 else None
    if sampler:
        sampler.start()
    l2_flush(flush_buf)
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    hold_stream()            # before e0: the host enqueues the graphs while the GPU spins
    wall0 = time.time()
    e0.record(stream)
    for _ in range(full):
        g_full.replay()
    if g_rem is not None:
        g_rem.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier()
    elapsed_ms = e0.elapsed_time(e1)
    clocks = sampler.stop(wall0, wall1) if sampler else None
    assert int(status.item()) == 0, "device status %d" % int(status.item())

    tokens = T * K
    job_ms, job_tokens = reduce_timing(elapsed_ms, tokens, dev)
    value = job_tokens / (job_ms / 1e3)
    nbytes = kv_algorithmic_bytes(T, 0, c0.Dv, c0.Dk)
    per_launch_s = elapsed_ms / 1e3 / K
    achieved = nbytes / per_launch_s / 1e9
    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs", 6800.0)
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    traffic, traffic_state = profiled_traffic()

    result = None
    if rank == 0:
        del kv, cos, sin, index, calls, graphs, g_full, g_rem
        torch.cuda.empty_cache()
        # the extras first: run after the two-stream staged loop, the decode
        # workload's 4096-call graph measured ~0.15 us per call slower
        extras = None if args.no_extras else run_extras(dev, kvr, flush_buf, peak)
        e2e = e2e_prefill(args, cases, gamma, ckv, kc, dev, kvr)
        cpu_tps, n_seq, cpu_s = cpu_oracle_baseline(args.cpu_seconds, c0)
        all_cores = cpu_oracle_all_cores(max(1.0, args.cpu_seconds / 2), c0)
        in_mb = R * T * ((c0.Dv + c0.Dk) * 2 + 4 * c0.Dk + 8) / 1e6
        result = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": job_ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD,
                       "step": "one kv_rmsnorm_rope_cache call on one 32768-token prefill batch",
                       "l2": "inputs larger than L2: steps rotate over %d input sets (%.0f MB > %.0f MB L2)"
                             % (R, in_mb, l2 / 1e6),
                       "launch": "CUDA graph replays of back-to-back calls (%d x %d-step graph + %d-step "
                                 "graph, each replayed once untimed first; a 1 ms device spin before the start "
                                 "event hides the host's launch latency)" % (full, G, rem),
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "hbm_gbs": achieved,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                         else peak_src,
                         "kernel": "kv_bulk_kernel", "bytes_per_launch": nbytes, "launch_us": per_launch_s * 1e6,
                         "traffic_source": PROFILE_SUMMARY.replace(ROOT + "/", "") if traffic else traffic_state},
            "cpu_baseline": {"value": cpu_tps, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": "%d whole 4096-token sequences of the prefill batch (%.1f s, float64 "
                                       "NumPy, one process)" % (n_seq, cpu_s),
                             "all_cores": None if all_cores is None else {
                                 "value": all_cores[0], "unit": UNIT, "cores": all_cores[1],
                                 "sample": "%d spawned processes, one per host core, %d sequences in %.1f s"
                                           % all_cores[1:]}},
            "e2e": e2e,
            "gpu_launches": K,
            "clocks": clocks,
            "extras": extras,
        }
    if world > 1:
        dist.destroy_process_group()
    return result


def e2e_prefill(args, cases, gamma, ckv, kc, dev, kvr):
    """Same metric through the public API with the inputs in pinned host
    memory: per step one host->device copy of the packed batch, the call, and
    a device->host read of the status word, all enqueued by one C call
    (kv_rmsnorm_rope_cache_staged). Steps alternate between two staging
    buffers on two streams, so that a step's call overlaps the next step's
    copy; timed over the K steps."""
    import torch
    R = len(cases)
    c0 = cases[0]
    kvb = c0.kv.numel() * 2
    csb = c0.cos.numel() * 2
    ixb = c0.index.numel() * 8
    blob = kvb + 2 * csb + ixb
    host = torch.empty(R, blob, dtype=torch.uint8).pin_memory()
    for i, c in enumerate(cases):
        host[i, :kvb] = c.kv.reshape(-1).view(torch.uint8)
        host[i, kvb:kvb + csb] = c.cos.reshape(-1).view(torch.uint8)
        host[i, kvb + csb:kvb + 2 * csb] = c.sin.reshape(-1).view(torch.uint8)
        host[i, kvb + 2 * csb:] = c.index.reshape(-1).view(torch.uint8)
    K = args.steps
    st_host = torch.zeros(K, dtype=torch.int32).pin_memory()
    streams = [torch.cuda.Stream(device=dev) for _ in range(2)]
    lanes = []
    for _ in range(2):
        stage = torch.empty(blob, dtype=torch.uint8, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        call = kvr.prepare_kv_rmsnorm_rope_cache(
            stage[:kvb].view(torch.bfloat16).view(c0.kv.shape), gamma,
            stage[kvb:kvb + csb].view(torch.bfloat16).view(c0.cos.shape),
            stage[kvb + csb:kvb + 2 * csb].view(torch.bfloat16).view(c0.sin.shape),
            stage[kvb + 2 * csb:].view(torch.int64), ckv, kc, cache_mode="PA_BSND", eps=1e-6, dev_status=status)
        lanes.append((call.staged, stage.data_ptr(), stage, status, call))
    host_ptr = [host[i].data_ptr() for i in range(R)]
    st_ptr = st_host.data_ptr()
    sids = [s_.cuda_stream for s_ in streams]

    def one(i, k):
        staged, stage_ptr = lanes[k % 2][0], lanes[k % 2][1]
        staged(host_ptr[i], stage_ptr, blob, st_ptr + 4 * k, sids[k % 2])

    for w in range(max(args.warmup, 3)):
        one(w % R, w % 2)
    torch.cuda.synchronize()
    main = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(main)
    for s_ in streams:
        s_.wait_event(e0)
    for k in range(K):
        one(k % R, k)
    for s_ in streams:
        done = torch.cuda.Event()
        done.record(s_)
        main.wait_event(done)
    e1.record(main)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    assert int(st_host.max()) == 0
    return {"value": c0.T * K / wall, "unit": UNIT, "h2d_bytes_per_step": blob, "d2h_bytes_per_step": 4,
            "device_ms": e0.elapsed_time(e1), "wall_ms": wall * 1e3,
            "how": "kv_rmsnorm_rope_cache_staged per step: packed pinned H2D copy, the call, status D2H; "
                   "two staging buffers on two streams, synchronised after the K steps"}


def hold_stream(ms=1.0):
    """Keep the current stream busy for about `ms` milliseconds (a device-side
    spin, no memory traffic), so that the host has enqueued what follows
    before the GPU reaches it: the start event then times the GPU work, not
    the host's graph-launch latency."""
    import torch
    torch.cuda._sleep(int(ms * 2e6))   # cycles at ~2 GHz


def time_graph(calls, n_calls, stream, reps=3):
    """Average duration of one call when n_calls calls (cycling through
    `calls`) run back to back as one CUDA graph replay (after one untimed
    replay); the median over `reps` timed replays."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n_calls):
            calls[i % len(calls)]()
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        hold_stream()
        e0.record(stream)
        g.replay()
        e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) / n_calls)
    return statistics.median(ts)


def run_extras(dev, kvr, flush_buf, peak):
    """The other workloads, each as {"us": microseconds per call, "frac":
    algorithmic bytes / time / measured HBM peak}: back-to-back calls in a
    CUDA graph over input sets that together exceed L2."""
    import torch

    from attention_prologue_kv_gb300 import workloads as wl
    out = {}
    stream = torch.cuda.current_stream()
    flush = lambda: l2_flush(flush_buf)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    def rec(us, nbytes):
        return {"us": round(us, 3), "frac": round(nbytes / (us / 1e6) / 1e9 / peak, 4)}

    # in-process copy references (16-byte vectorised device copy): 2 x 512 MB, and
    # the prefill's size (42 MB read + 42 MB written) back to back over rotating sources
    src = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    dst = torch.empty_like(src)
    _, best = time_each(lambda: kvr.device_copy(dst, src), 10, flush, stream)
    out["copy_1GB"] = rec(best * 1e3, 2 * src.numel())
    del src, dst
    half = 84149248 // 2 // 16 * 16
    n_pairs = int(2 * l2 // (2 * half)) + 2
    bufs = [(torch.empty(half, dtype=torch.uint8, device=dev), torch.empty(half, dtype=torch.uint8, device=dev))
            for _ in range(n_pairs)]
    calls = [lambda b=b: kvr.device_copy(b[1], b[0]) for b in bufs]
    out["copy_84MB"] = rec(time_graph(calls, 8 * len(calls), stream) * 1e3, 2 * half)
    del bufs, calls

    def nsets(bytes_per_set):
        return max(3, int(2 * l2 // bytes_per_set) + 1)

    # decode: 256-token batches, 512 sets rotated (186 MB)
    sets = wl.decode_paged_sets(512, seed=1002)
    d0, d1 = sets["d0"], sets["d1"]
    ckv = torch.zeros(d0, d1, 1, 512, dtype=torch.bfloat16, device=dev)
    kc = torch.zeros(d0, d1, 1, 64, dtype=torch.bfloat16, device=dev)
    kv, cs, sn, ix = (sets[k].to(dev) for k in ("kv", "cos", "sin", "index"))
    gamma = sets["gamma"].to(dev)
    calls = [kvr.prepare_kv_rmsnorm_rope_cache(kv[i], gamma, cs[i], sn[i], ix[i], ckv, kc, cache_mode="PA_BSND")
             for i in range(512)]
    skips = (sets["index"] == -1).sum(dim=1).tolist()
    nbytes = statistics.fmean(kv_algorithmic_bytes(256 - s, s) for s in skips)
    out["decode_paged"] = rec(time_graph(calls, 4096, stream) * 1e3, nbytes)
    del calls, kv, cs, sn, ix, ckv, kc, sets

    def kv_workload(make, seeds, params_ready=False):
        cases = [make(seed=s) for s in seeds]
        c0 = cases[0]
        ckv = torch.zeros(c0.cache_shapes()[0], dtype=wl.code_torch_dtype(c0.ckv_dtype), device=dev).view(
            wl.TORCH_DTYPES[c0.ckv_dtype])
        kc = torch.zeros(c0.cache_shapes()[1], dtype=wl.code_torch_dtype(c0.k_dtype), device=dev).view(
            wl.TORCH_DTYPES[c0.k_dtype])
        calls = []
        for c in cases:
            calls.append(kvr.prepare_kv_rmsnorm_rope_cache(
                c.kv.to(dev), c.gamma.to(dev), c.cos.to(dev), c.sin.to(dev), c.index.to(dev), ckv, kc,
                cache_mode=c.mode, eps=c.eps, ckv_scale=None if c.ckv_scale is None else c.ckv_scale.to(dev),
                params_ready=params_ready))
        act = c0.active_tokens()
        nbytes = kv_algorithmic_bytes(act, c0.T - act, c0.Dv, c0.Dk,
                                      ckv_bytes=1 if c0.ckv_dtype != "bf16" else 2,
                                      scale_bytes=0 if c0.ckv_scale is None else 4 * c0.ckv_scale.numel())
        return rec(time_graph(calls, max(8 * len(calls), 48), stream) * 1e3, nbytes)

    out["quant_fp8"] = kv_workload(wl.quant_fp8, [1004 + 7919 * i for i in range(nsets(4096 * 1416))])
    # the same with params_ready: gamma and the scales read before the dependency wait
    out["quant_fp8_params_ready"] = kv_workload(wl.quant_fp8, [1004 + 7919 * i for i in range(nsets(4096 * 1416))],
                                                params_ready=True)
    out["tiny_norm"] = kv_workload(wl.tiny_norm, [1001])

    # QSA prepare: default form, rotate-half on the first Dr channels, params_ready,
    # and the concat-output form (past block keys [N, Bp, Di] copied into a fresh output first)
    qs = [wl.qsa_prepare_workload(seed=1005 + 7919 * i) for i in range(nsets(17.3e6))]
    q0 = qs[0]
    nb = q0.completed_blocks()
    qbytes = qsa_algorithmic_bytes(nb, q0.N, q0.kbs, q0.Di, q0.Dr)
    bk = torch.zeros(q0.N, q0.Bcap, q0.Di, dtype=torch.bfloat16, device=dev)
    d = lambda t: t.to(dev)
    Bp = int(max(max(p_ // q.kbs for p_ in q.meta["past"]) for q in qs))
    past_bk = torch.zeros(q0.N, Bp, q0.Di, dtype=torch.bfloat16, device=dev)
    qsa_args = [(d(q.raw), bk, d(q.key_length), d(q.rope_cos), d(q.rope_sin), d(q.k_norm_weight),
                d(q.past_raw), d(q.past_rope), q.kbs, q.eps) for q in qs]
    for name, kw, extra in (
            ("qsa_prepare", {}, lambda q: 0),
            ("qsa_prepare_half_first", dict(rope_layout="half_first"), lambda q: 0),
            ("qsa_prepare_params_ready", dict(params_ready=True), lambda q: 0),
            ("qsa_prepare_concat", dict(past_block_index_keys=past_bk),
             lambda q: 2 * q.Di * 2 * sum(min(Bp, p_ // q.kbs) for p_ in q.meta["past"]))):
        calls = [lambda a=a, kw=kw: kvr.qsa_prepare(*a, **kw) for a in qsa_args]
        extra_mean = sum(extra(q) for q in qs) / len(qs)   # copied rows differ between sets
        out[name] = rec(time_graph(calls, 8 * len(calls), stream) * 1e3, qbytes + extra_mean)
    del past_bk, qsa_args, calls, qs, bk

    # the same kernel at 8x the new tokens (32 x 16384): separates its fixed
    # per-call latency from its streaming rate
    qb = [wl.make_qsa_case("qsa_prepare_L16384", 32, 16384, Di=128, Dr=64, kbs=64, seed=1105 + 7919 * i,
                           past_max=8192, Bcap=400) for i in range(3)]
    bkb = torch.zeros(32, 400, 128, dtype=torch.bfloat16, device=dev)
    calls = []
    for q in qb:
        a = (d(q.raw), bkb, d(q.key_length), d(q.rope_cos), d(q.rope_sin), d(q.k_norm_weight),
             d(q.past_raw), d(q.past_rope), q.kbs, q.eps)
        calls.append(lambda a=a: kvr.qsa_prepare(*a))
    out["qsa_prepare_L16384"] = rec(time_graph(calls, 8 * len(calls), stream) * 1e3,
                                    qsa_algorithmic_bytes(qb[0].completed_blocks(), 32, 64, 128, 64))
    del qb, calls, bkb

    # DynamicQuant of q^N for one decode step (256 tokens x 128 heads x 512), default and exact
    qs = [wl.dynamic_quant_decode(seed=1006 + 7919 * i) for i in range(nsets(256 * 128 * 512 * 2))]
    rows, H = qs[0].numel() // qs[0].shape[-1], qs[0].shape[-1]
    outs = [(q.to(dev), torch.empty(q.shape, dtype=torch.int8, device=dev),
             torch.empty(q.shape[:-1] + (1,), dtype=torch.float32, device=dev)) for q in qs]
    for name, exact in (("dynamic_quant_decode", False), ("dynamic_quant_decode_exact", True)):
        calls = [lambda o=o, e=exact: kvr.dynamic_quant(*o, exact=e) for o in outs]
        out[name] = rec(time_graph(calls, 8 * len(calls), stream) * 1e3, dq_algorithmic_bytes(rows, H))
    torch.cuda.synchronize()
    return out


# ---------------------------------------------------------------------------
# Reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    """The oracle as it stands on the prefill workload: each step runs it over
    a bounded sample of one prefill batch (whole sequences; all 8 when the
    W + K steps fit in about two minutes)."""
    cases = prefill_sets(2)
    c0 = cases[0]
    seqs = [_oracle_seqs(c, c.Bkv) for c in cases]
    import numpy as np

    import oracle
    ckv = np.full((c0.d0, c0.d1, c0.Dv), 0x7FBF, dtype=np.uint16)
    kc = np.full((c0.d0, c0.d1, c0.Dk), 0x7FBF, dtype=np.uint16)

    def step(i, n_seq):
        ss, gamma = seqs[i % len(seqs)]
        for kv, cos, sin, idx in ss[:n_seq]:
            oracle.ref_kv_rmsnorm_rope_cache(kv, gamma, cos, sin, idx, ckv, kc, Dv=c0.Dv, mode="PA_BSND", eps=1e-6)

    t = time.perf_counter()
    step(0, 1)
    t_seq = time.perf_counter() - t
    budget = 120.0
    n_seq = int(max(1, min(c0.Bkv, budget / ((args.steps + args.warmup) * t_seq))))
    for w in range(args.warmup):
        step(w, n_seq)
    t0 = time.perf_counter()
    for k in range(args.steps):
        step(k, n_seq)
    el = time.perf_counter() - t0
    ntok = n_seq * c0.Skv
    value = ntok * args.steps / el
    sample = ("%d of the 8 sequences (%d of 32768 tokens) of a prefill batch per step, float64 NumPy oracle, "
              "one process" % (n_seq, ntok))
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "step": "oracle on a bounded sample of one "
                                                                           "prefill batch"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_only(args):
    """W + K launches of a single workload, timed per launch (no L2 flush, no
    graphs): a small, self-contained command for profilers."""
    import torch

    import attention_prologue_kv_gb300 as kvr
    from attention_prologue_kv_gb300 import workloads as wl
    from attention_prologue_kv_gb300.build import build
    build()
    dev = torch.device("cuda", 0)
    if args.only in ("qsa_prepare", "qsa_prepare_params_ready"):
        # the input sets the extras rotate through (together larger than L2)
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        qs = [wl.qsa_prepare_workload(seed=1005 + 7919 * i) for i in range(max(3, int(2 * l2 // 17.3e6) + 1))]
        bk = torch.zeros(qs[0].N, qs[0].Bcap, qs[0].Di, dtype=torch.bfloat16, device=dev)
        d = lambda t: t.to(dev)
        args_q = [(d(q.raw), bk, d(q.key_length), d(q.rope_cos), d(q.rope_sin), d(q.k_norm_weight),
                   d(q.past_raw), d(q.past_rope), q.kbs, q.eps) for q in qs]
        pr = args.only == "qsa_prepare_params_ready"
        it = iter(range(1 << 62))
        fn = lambda: kvr.qsa_prepare(*args_q[next(it) % len(args_q)], params_ready=pr)
    elif args.only in ("dynamic_quant_decode", "dynamic_quant_decode_exact"):
        q = wl.dynamic_quant_decode().to(dev)
        o = torch.empty(q.shape, dtype=torch.int8, device=dev)
        sc = torch.empty(q.shape[:-1] + (1,), dtype=torch.float32, device=dev)
        ex = args.only == "dynamic_quant_decode_exact"
        fn = lambda: kvr.dynamic_quant(q, o, sc, exact=ex)
    elif args.only == "decode_paged":
        # the decode batches the extras rotate through (512 sets, larger than L2)
        sets = wl.decode_paged_sets(512, seed=1002)
        ckv = torch.zeros(sets["d0"], sets["d1"], 1, 512, dtype=torch.bfloat16, device=dev)
        kc = torch.zeros(sets["d0"], sets["d1"], 1, 64, dtype=torch.bfloat16, device=dev)
        kv, cs, sn, ix = (sets[k].to(dev) for k in ("kv", "cos", "sin", "index"))
        gamma = sets["gamma"].to(dev)
        calls = [kvr.prepare_kv_rmsnorm_rope_cache(kv[i], gamma, cs[i], sn[i], ix[i], ckv, kc, cache_mode="PA_BSND")
                 for i in range(512)]
        it = iter(range(1 << 62))
        fn = lambda: calls[next(it) % len(calls)]()
    else:
        # prefill: the benchmark's rotation of input sets (larger than L2); others: one set
        cases = prefill_sets(ROTATION) if args.only == "prefill_paged" else [getattr(wl, args.only)()]
        case = cases[0]
        ckv = torch.zeros(case.cache_shapes()[0], dtype=wl.code_torch_dtype(case.ckv_dtype), device=dev).view(
            wl.TORCH_DTYPES[case.ckv_dtype])
        kc = torch.zeros(case.cache_shapes()[1], dtype=wl.code_torch_dtype(case.k_dtype), device=dev).view(
            wl.TORCH_DTYPES[case.k_dtype])
        calls = [kvr.prepare_kv_rmsnorm_rope_cache(
            c.kv.to(dev), case.gamma.to(dev), c.cos.to(dev), c.sin.to(dev), c.index.to(dev), ckv, kc,
            cache_mode=c.mode, eps=c.eps, ckv_scale=None if c.ckv_scale is None else c.ckv_scale.to(dev))
            for c in cases]
        it = iter(range(1 << 62))
        fn = lambda: calls[next(it) % len(calls)]()
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    if args.profile_range:
        cudart = torch.cuda.cudart()
        if args.profile_graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for _ in range(args.steps):
                    fn()
            g.replay()
            torch.cuda.synchronize()
            cudart.cudaProfilerStart()
            g.replay()
            torch.cuda.synchronize()
            cudart.cudaProfilerStop()
            return {"only": args.only, "launches": args.warmup + 2 * args.steps, "range": args.steps,
                    "graph": True}
        cudart.cudaProfilerStart()
        for _ in range(args.steps):
            fn()
        cudart.cudaProfilerStop()
        torch.cuda.synchronize()
        return {"only": args.only, "launches": args.warmup + args.steps, "range": args.steps}
    stream = torch.cuda.current_stream()
    ts = []
    for _ in range(args.steps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    return {"only": args.only, "launches": args.warmup + args.steps, "us_median": statistics.median(ts),
            "us_min": min(ts)}


def main(argv=None):
    args = parse_args(argv)
    rank, world, _ = dist_env()
    if args.only:
        print(json.dumps(run_only(args)), flush=True)
        return 0
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0
    if args.extras_only:
        import torch

        import attention_prologue_kv_gb300 as kvr
        from attention_prologue_kv_gb300.build import build
        build()
        dev = torch.device("cuda", 0)
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        flush_buf = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
        peak = measured_peaks().get("hbm_gbs", 6800.0)
        print(json.dumps({"extras": run_extras(dev, kvr, flush_buf, peak)}), flush=True)
        return 0
    res = run_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
