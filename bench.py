#!/usr/bin/env python
"""Benchmark of the exact-attention hot path on one GB300 (replicas on N GPUs).

One step = one pass of the whole path on one synthetic batch:
  * prefill: causal MHA, B=4, Hq=Hkv=32, N=4096, d=128, bf16 (tensor-core kernel);
  * decode: paged split-KV, batch 8, Hq=32, Hkv=8, d=128, contexts U[1024, 65536]
    (seed 4), 16-token pages (decode-partials kernel + merge kernel).
``value`` is prefill causal-adjusted TFLOP/s (4*B*Hq*N^2*d / 2 per step) summed
over ranks; decode KV GB/s is reported beside it. Inputs are resident in HBM
when timing starts. Before every timed launch L2 is flushed: a 256 MB buffer
is written, then a second 256 MB buffer is read, so the launch finds neither
its inputs nor dirty lines (whose write-back it would otherwise pay) in L2.
``e2e`` repeats the step through the same public API from pinned host buffers,
host<->device copies included: every step copies its inputs in and its outputs
out, double-buffered on three streams so that one step's copies overlap the
neighbouring steps' kernels and copies (the host link, not the kernels, sets it).

``--impl reference`` times the fp64 CPU oracle on the host cores instead, on a
bounded sample of the same prefill workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill attention TFLOP/s & decode KV GB/s, % of GB300 roofline (1 GPU)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--num-splits", type=int, default=0, help="decode splits (0 = library heuristic)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sparse", action="store_true",
                    help="skip the block-sparse, paged, masked and FP8 prefill and backward measurements "
                         "(outside the step)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the cpu_baseline sample")
    ap.add_argument("--cpu-leg-seconds", type=float, default=6.0,
                    help="budget of the oracle timed beside each of the other legs (decode, long GQA, varlen)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the long-context GQA and ragged varlen prefill measurements (outside the step)")
    ap.add_argument("--profile-once", action="store_true",
                    help="one launch each of prefill, decode, block-sparse, paged, masked and FP8 prefill "
                         "and backward on the bench workloads, then exit (for ncu)")
    return ap.parse_args()


KERNEL_SOURCES = {
    "prefill_tc_kernel<128>": ["prefill_tc.cu", "sm100_primitives.cuh", "device_common.cuh", "fattn_internal.h"],
    "decode_kernel<128, page16>": ["decode.cu", "device_common.cuh", "fattn_internal.h"],
}
KERNEL_SOURCES["prefill_tc_kernel<128, sparse>"] = KERNEL_SOURCES["prefill_tc_kernel<128>"]
KERNEL_SOURCES["prefill_tc_kernel<128, paged>"] = KERNEL_SOURCES["prefill_tc_kernel<128>"]
KERNEL_SOURCES["prefill_tc_kernel<128, masked>"] = KERNEL_SOURCES["prefill_tc_kernel<128>"]
KERNEL_SOURCES["prefill_tc_kernel<128, fp8>"] = KERNEL_SOURCES["prefill_tc_kernel<128>"]
KERNEL_SOURCES["prefill_tc_kernel<128>, long GQA"] = KERNEL_SOURCES["prefill_tc_kernel<128>"]
KERNEL_SOURCES["prefill_tc_kernel<64>, varlen"] = KERNEL_SOURCES["prefill_tc_kernel<128>"]
KERNEL_SOURCES["bwd_dkdv_kernel<128>"] = ["backward.cu", "sm100_primitives.cuh", "device_common.cuh", "fattn_internal.h"]
KERNEL_SOURCES["bwd_dq_kernel<128>"] = KERNEL_SOURCES["bwd_dkdv_kernel<128>"]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from profiles/dram_traffic.md, or None when the
    kernel's sources changed since that capture (or none was recorded)."""
    import hashlib
    csrc = os.path.join(ROOT, "exact_tiled_attention_fattn_gb300", "csrc")
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.md")) as fh:
            for line in fh:
                cells = [c.strip() for c in line.strip().strip("|").split("|")]
                if len(cells) == 3 and cells[0] == kernel and cells[2] == h.hexdigest()[:16]:
                    return float(cells[1])
    except OSError:
        pass
    return None


def max_over_ranks(vals, world: int, device=None):
    """Each value's maximum over the ranks (the slowest replica sets the step time).
    One rank: the values unchanged. Works on any process group backend (NCCL on the
    GPU machine with a CUDA device, gloo in the CPU tests with device=None)."""
    vals = [float(v) for v in vals]
    if world <= 1:
        return vals
    import torch
    import torch.distributed as dist
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu().tolist()]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        # samples under load: the upper half by power
        thr = sorted(power)[len(power) // 2] if power else 0
        loaded = [s for s, p in zip(sm, power) if p >= thr] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- workloads
def make_workloads():
    from exact_tiled_attention_fattn_gb300 import inputs
    pre = inputs.causal_mha_config()
    dec = inputs.paged_decode_config()
    return pre, dec


def local_global_mask(nb: int, window: int):
    """Block mask [1, nb, nb]: each query block keeps its `window` nearest key
    blocks at or below the diagonal and the first block."""
    import numpy as np
    m = np.zeros((1, nb, nb), np.uint8)
    for i in range(nb):
        m[0, i, max(0, i - window + 1): i + 1] = 1
        m[0, i, 0] = 1
    return m


def block_sparse_flops(mask, B: int, H: int, d: int, blk: int = 128) -> float:
    """Causal work in the kept blocks, counted like the dense convention: a
    block below the diagonal is blk^2 (q, k) pairs, a diagonal block blk^2 / 2."""
    import numpy as np
    m = np.tril(mask[0])
    pairs = float(np.sum(m)) * blk * blk - float(np.trace(m)) * blk * blk / 2
    return 4.0 * d * pairs * B * H


def block_sparse_leg(fattn, pre, q, k, v, o, lse, flush, stream, peaks):
    """Block-sparse prefill on the bench's causal MHA inputs: a local (3 blocks)
    + global (first block) mask, and the all-kept causal mask, which does the
    dense kernel's work through the sparse path."""
    import numpy as np
    import torch
    B, N, H, d = pre.q.shape
    nb = N // 128
    res = {"workload": f"causal MHA B={B} Hq=Hkv={H} N={N} d={d}, 128x128 blocks, one mask for all heads"}
    for name, window in (("local3_global", 3), ("all_causal_blocks", nb)):
        mh = local_global_mask(nb, window)
        mt = torch.from_numpy(mh).to(q.device)
        run = lambda: fattn.fwd_block_sparse(q, k, v, mt, causal=True, scale=pre.scale, out=o, lse=lse)
        for _ in range(3):
            flush()
            run()
        ts = []
        for _ in range(10):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        t = statistics.median(ts)
        fl = block_sparse_flops(mh, B, H, d)
        tf = fl / (t * 1e-3) / 1e12
        res[name] = {"ms": t, "kept_block_fraction": float(np.tril(mh[0]).sum()) / (nb * (nb + 1) / 2),
                     "tflops": tf, "frac_of_bf16_peak": tf / peaks["bf16_tflops"]}
    res["local3_global"]["traffic"] = recorded_traffic("prefill_tc_kernel<128, sparse>")
    return res


def paged_prefill_workload():
    """Chunked prefill: B=4, Hq=32, Hkv=8, d=128, 16-token pages, contexts U[4096, 16384]
    (seed 710), the last 2048 positions of each context as the chunk's queries."""
    from exact_tiled_attention_fattn_gb300 import inputs
    return inputs.prefill_paged(710, 4, 32, 8, 128, 16, (4096, 16384), 2048, 16384, causal=True)


def paged_prefill_leg(fattn, flush, stream, peaks, dev):
    """fattn_fwd_paged on the chunked-prefill workload (10 launches, median)."""
    import torch
    x = paged_prefill_workload()
    args = [t.to(dev) for t in (x.q, x.kcache, x.vcache, x.block_table, x.seqlens_k, x.cu_seqlens_q)]
    o = torch.empty_like(args[0])
    lse = torch.empty((x.hq, args[0].shape[0]), dtype=torch.float32, device=dev)
    run = lambda: fattn.fwd_paged(*args, max(x.lengths_q), causal=True, scale=x.scale, out=o, lse=lse)
    for _ in range(3):
        flush()
        run()
    ts = []
    for _ in range(10):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    t = statistics.median(ts)
    tf = x.flops() / (t * 1e-3) / 1e12
    kv = 2 * sum(x.lengths_k) * x.hkv * x.d * 2
    return {"workload": "chunked prefill B=4 Hq=32 Hkv=8 d=128, 16-token pages, contexts U[4096,16384] seed 710 "
                        f"({sum(x.lengths_k)} tokens), 2048-query chunks, causal bottom-right",
            "ms": t, "tflops": tf, "frac_of_bf16_peak": tf / peaks["bf16_tflops"], "flops": x.flops(),
            "kv_bytes": kv, "traffic": recorded_traffic("prefill_tc_kernel<128, paged>")}


def backward_leg(fattn, pre, q, k, v, o, lse, flush, stream, peaks, dev):
    """fattn_bwd on the prefill workload (dO ~ N(0, 1), seed 5; O and lse from fattn_fwd), 10 launches, median.
    Work convention: 2.5 x the forward's FLOPs (five products of the forward's size, the usual count)."""
    import torch
    g = torch.Generator("cpu").manual_seed(5)
    do = torch.randn(pre.q.shape, generator=g).to(torch.bfloat16).to(dev)
    fattn.fwd(q, k, v, causal=True, scale=pre.scale, out=o, lse=lse)
    B, N, Hq, _ = pre.q.shape
    ws = torch.empty(fattn.bwd_workspace_size(B, Hq, N), dtype=torch.uint8, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    run = lambda: fattn.bwd(q, k, v, o, lse, do, causal=True, scale=pre.scale, dq=dq, dk=dk, dv=dv, workspace=ws)
    for _ in range(3):
        flush()
        run()
    ts = []
    for _ in range(10):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    t = statistics.median(ts)
    fl = 2.5 * pre.flops()
    tf = fl / (t * 1e-3) / 1e12
    return {"workload": "backward of the causal MHA prefill B=4 Hq=Hkv=32 N=4096 d=128 (dQ pass, which also forms "
                        "the per-row vectors, then dK/dV pass)", "ms": t, "tflops": tf,
            "frac_of_bf16_peak": tf / peaks["bf16_tflops"], "flops": fl, "launches": 2,
            "traffic": {"bwd_dkdv_kernel<128>": recorded_traffic("bwd_dkdv_kernel<128>"),
                        "bwd_dq_kernel<128>": recorded_traffic("bwd_dq_kernel<128>")}}


def _time_launches(run, flush, stream, n=10):
    import torch
    for _ in range(3):
        flush()
        run()
    ts = []
    for _ in range(n):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def alibi_mask(N: int, dev):
    """One shared bf16 additive mask [1, 1, N, N]: M[i, j] = -0.01 (i - j)."""
    import torch
    i = torch.arange(N, dtype=torch.float32, device=dev)
    return (-0.01 * (i[:, None] - i[None, :])).to(torch.bfloat16)[None, None].contiguous()


def masked_leg(fattn, pre, q, k, v, o, lse, flush, stream, peaks, dev):
    """fattn_fwd_masked on the prefill inputs with one shared ALiBi-style bias, causal."""
    m = alibi_mask(pre.q.shape[1], dev)
    t = _time_launches(lambda: fattn.fwd_masked(q, k, v, m, causal=True, scale=pre.scale, out=o, lse=lse), flush,
                       stream)
    tf = pre.flops() / (t * 1e-3) / 1e12
    return {"workload": "causal MHA B=4 Hq=Hkv=32 N=4096 d=128 + one shared bf16 bias M[i,j] = -0.01 (i - j)",
            "ms": t, "tflops": tf, "frac_of_bf16_peak": tf / peaks["bf16_tflops"],
            "traffic": recorded_traffic("prefill_tc_kernel<128, masked>")}


def fp8_leg(fattn, pre, flush, stream, peaks, dev):
    """fattn_fwd_fp8 on E4M3 inputs of the prefill workload's shape (seed 1, per-tensor descales)."""
    import torch
    from exact_tiled_attention_fattn_gb300 import inputs
    B, N, Hq, d = pre.q.shape
    x = inputs.prefill_fp8(1, B, N, Hq, pre.hkv, d, True)
    q8, k8, v8 = x.q8.to(dev), x.k8.to(dev), x.v8.to(dev)
    o = torch.empty(q8.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    t = _time_launches(lambda: fattn.fwd_fp8(q8, k8, v8, x.q_descale, x.k_descale, x.v_descale, causal=True,
                                             scale=x.scale, out=o, lse=lse), flush, stream)
    tf = x.flops() / (t * 1e-3) / 1e12
    peak8, src8 = fp8_gemm_peak(dev)
    if peak8 is None:
        peak8 = 2.0 * peaks["bf16_tflops"]   # the measured bf16 peak x the nominal fp8 : bf16 ratio (4.5 : 2.25)
        src8 = f"measured bf16_tflops x 2 (nominal fp8/bf16 ratio; the FP8 GEMM could not be timed: {src8})"
    return {"workload": "causal MHA B=4 Hq=Hkv=32 N=4096 d=128, E4M3 q, k, v (per-tensor descales), bf16 O",
            "ms": t, "tflops": tf, "peak_fp8_tflops": peak8,
            "peak_source": src8, "frac_of_fp8_peak": tf / peak8,
            "launches": 1, "traffic": recorded_traffic("prefill_tc_kernel<128, fp8>")}


def fp8_gemm_peak(dev, n: int = 8192, reps: int = 10):
    """Dense E4M3 tensor throughput measured on this GPU the way the bf16 peak is: a library
    GEMM (cuBLASLt through torch._scaled_mm, per-tensor scales, bf16 out) of n^3, best of
    `reps`, CUDA events. Returns (TFLOP/s, how) or (None, why not)."""
    import torch
    try:
        g = torch.Generator(device=dev).manual_seed(0)
        a = torch.randn((n, n), device=dev, generator=g).to(torch.float8_e4m3fn)
        b = torch.randn((n, n), device=dev, generator=g).to(torch.float8_e4m3fn).t()   # column-major operand
        one = torch.ones((), dtype=torch.float32, device=dev)
        mm = lambda: torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        for _ in range(3):
            mm()
        best = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            mm()
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12, (f"measured: torch._scaled_mm E4M3 {n}^3 (cuBLASLt, per-tensor "
                                                      f"scales, bf16 out), best of {reps}, CUDA events")
    except Exception as e:  # noqa: BLE001 - report why the GEMM could not be timed
        return None, f"{type(e).__name__}: {str(e)[:120]}"


def cpu_baseline_rows(x, seconds: float, what: str, chunk: int = 64):
    """Time the fp64 oracle on random chunks of query rows of a causal prefill workload
    (dense [B, N, H, d] or varlen [T, H, d] with cu_seqlens), on the host cores."""
    import numpy as np
    from oracle import attention as orc
    rng = np.random.default_rng(0)
    varlen = x.cu_seqlens is not None
    d = x.q.shape[-1]
    if varlen:
        cu = [int(c) for c in x.cu_seqlens]
        lens = [cu[b + 1] - cu[b] for b in range(len(cu) - 1)]
        H = x.q.shape[1]
    else:
        B, N, H = x.q.shape[0], x.q.shape[1], x.q.shape[2]
        lens = [N] * B
    done_rows, flops, t_used, groups = 0, 0.0, 0.0, 0
    while t_used < seconds:
        b, h = int(rng.integers(len(lens))), int(rng.integers(H))
        n = min(chunk, lens[b])
        rows = np.sort(rng.choice(lens[b], size=n, replace=False))
        smp = np.stack([np.full(n, b), np.full(n, h), rows], axis=1)
        t0 = time.perf_counter()
        if varlen:
            orc.attn_fwd_rows(x.q, x.k, x.v, x.scale, True, smp, cu_seqlens=x.cu_seqlens)
        else:
            orc.attn_fwd_rows(x.q, x.k, x.v, x.scale, True, smp)
        t_used += time.perf_counter() - t0
        flops += float(np.sum(4.0 * d * (rows + 1)))      # causal: row i sees i+1 keys
        done_rows += n
        groups += 1
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": flops / t_used / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{done_rows} query rows ({groups} random (sequence, head) groups of up to {chunk} rows) "
                      f"of the {what}, fp64 numpy (BLAS threads = cores), {t_used:.1f} s"}


def prefill_config_leg(fattn, x, what, kernel, flush, stream, peaks, dev, cpu_seconds):
    """fattn_fwd on one more prefill workload (10 launches, median, L2 flushed before each),
    with its roofline against the measured bf16 burst peak and the oracle timed beside it."""
    import torch
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    o = torch.empty_like(q)
    if x.cu_seqlens is not None:
        cu = x.cu_seqlens.to(dev)
        lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=dev)
        run = lambda: fattn.fwd(q, k, v, causal=True, scale=x.scale, cu_seqlens=cu, max_seqlen=x.max_seqlen,
                                out=o, lse=lse)
    else:
        lse = torch.empty((q.shape[0], q.shape[2], q.shape[1]), dtype=torch.float32, device=dev)
        run = lambda: fattn.fwd(q, k, v, causal=True, scale=x.scale, out=o, lse=lse)
    t = _time_launches(run, flush, stream)
    tf = x.flops() / (t * 1e-3) / 1e12
    res = {"workload": what, "ms": t, "tflops": tf, "flops": x.flops(),
           "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                        "frac": tf / peaks["bf16_tflops"], "traffic": recorded_traffic(kernel),
                        "peak_source": "measured bf16_tflops (burst)", "kernel": kernel}}
    del q, k, v, o, lse
    if cpu_seconds > 0:
        res["cpu_baseline"] = cpu_baseline_rows(x, cpu_seconds, what)
    return res


def cpu_baseline_decode(dec, seconds: float):
    """Time the fp64 oracle's paged decode on the host cores, one sequence of the decode
    workload at a time (in order) until the budget is spent; KV bytes read per second."""
    from oracle import attention as orc
    t_used, kv, seqs, toks = 0.0, 0.0, 0, 0
    for b in range(dec.batch):
        if t_used >= seconds:
            break
        sl = dec.seqlens[b:b + 1]
        t0 = time.perf_counter()
        orc.decode_paged(dec.q[b:b + 1], dec.kcache, dec.vcache, dec.block_table[b:b + 1], sl, dec.scale)
        t_used += time.perf_counter() - t0
        n = int(sl[0])
        kv += 2.0 * n * dec.hkv * dec.d * 2
        seqs += 1
        toks += n
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": kv / t_used / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{seqs} of the {dec.batch} decode sequences ({toks} context tokens, all {dec.hq} query "
                      f"heads), paged gather + fp64 definition in numpy, {t_used:.1f} s"}


def cpu_baseline_prefill(pre, seconds: float):
    """Time the fp64 oracle on sampled query rows of the prefill workload."""
    import numpy as np
    from oracle import attention as orc
    B, N, Hq, d = pre.q.shape
    rng = np.random.default_rng(0)
    done_rows, flops, t_used = 0, 0.0, 0.0
    chunk = 64
    heads = 0
    while t_used < seconds:
        b, h = int(rng.integers(B)), int(rng.integers(Hq))
        rows = np.sort(rng.choice(N, size=chunk, replace=False))
        smp = np.stack([np.full(chunk, b), np.full(chunk, h), rows], axis=1)
        t0 = time.perf_counter()
        orc.attn_fwd_rows(pre.q, pre.k, pre.v, pre.scale, True, smp)
        t_used += time.perf_counter() - t0
        flops += float(np.sum(4.0 * d * (rows + 1)))      # causal: row i sees i+1 keys
        done_rows += chunk
        heads += 1
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": flops / t_used / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{done_rows} query rows ({heads} random (b, head) pairs x {chunk} rows) of the "
                      f"B=4 H=32 N=4096 d=128 causal prefill, fp64 numpy (BLAS threads = cores), "
                      f"{t_used:.1f} s"}


def run_reference(args):
    """The oracle as it stands, on host cores, on bounded samples of the prefill workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    pre, _ = make_workloads()
    per_step = max(1.0, min(6.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_baseline_prefill(pre, per_step / 4)
    vals = [cpu_baseline_prefill(pre, per_step) for _ in range(args.steps)]
    v = statistics.median(x["value"] for x in vals)
    cb = dict(vals[-1])
    cb["value"] = v
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "ms_per_step": per_step * 1e3,
            "config": {"workload": "causal MHA prefill B=4 Hq=Hkv=32 N=4096 d=128 (oracle on sampled rows)",
                       "l2": "n/a (host)"},
            "cpu_baseline": cb,
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    import torch.distributed as dist
    from exact_tiled_attention_fattn_gb300 import build, fattn

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build.build()
    fattn.load_library()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    pre, dec = make_workloads()
    q, k, v = pre.q.to(dev), pre.k.to(dev), pre.v.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((pre.q.shape[0], pre.hq, pre.q.shape[1]), dtype=torch.float32, device=dev)
    dq, dk, dv = dec.q.to(dev), dec.kcache.to(dev), dec.vcache.to(dev)
    dbt, dsl = dec.block_table.to(dev), dec.seqlens.to(dev)
    S = args.num_splits or fattn.choose_num_splits(dec.batch, dec.hkv, dec.max_pages_per_seq)
    ws = torch.zeros(fattn.decode_workspace_size(dec.batch, dec.hq, dec.d, S), dtype=torch.uint8, device=dev)
    do = torch.empty_like(dq)
    dlse = torch.empty((dec.batch, dec.hq), dtype=torch.float32, device=dev)
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def flush():
        flush_w.zero_()
        flush_r.max()

    def prefill():
        fattn.fwd(q, k, v, causal=True, scale=pre.scale, out=o, lse=lse)

    def decode():
        fattn.decode_paged(dq, dk, dv, dbt, dsl, S, scale=dec.scale, out=do, lse=dlse, workspace=ws)

    if args.profile_once:
        from exact_tiled_attention_fattn_gb300 import inputs
        prefill()
        decode()
        if not args.no_sparse:  # one block-sparse launch: local (3 blocks) + global mask
            nb = pre.q.shape[1] // 128
            mt = torch.from_numpy(local_global_mask(nb, 3)).to(dev)
            fattn.fwd_block_sparse(q, k, v, mt, causal=True, scale=pre.scale, out=o, lse=lse)
            x = paged_prefill_workload()            # and one paged (chunked) prefill launch
            pa = [t.to(dev) for t in (x.q, x.kcache, x.vcache, x.block_table, x.seqlens_k, x.cu_seqlens_q)]
            fattn.fwd_paged(*pa, max(x.lengths_q), causal=True, scale=x.scale)
            fattn.fwd_masked(q, k, v, alibi_mask(pre.q.shape[1], dev), causal=True, scale=pre.scale)  # masked
            x8 = inputs.prefill_fp8(1, *pre.q.shape[:3], pre.hkv, pre.q.shape[3], True)  # and FP8
            fattn.fwd_fp8(x8.q8.to(dev), x8.k8.to(dev), x8.v8.to(dev), x8.q_descale, x8.k_descale, x8.v_descale,
                          causal=True, scale=x8.scale)
            do = torch.randn(q.shape, device=dev).to(torch.bfloat16)  # and one backward
            prefill()
            fattn.bwd(q, k, v, o, lse, do, causal=True, scale=pre.scale)
        if not args.no_configs:  # one long-context GQA and one varlen prefill launch
            xg = inputs.long_gqa_config()
            fattn.fwd(xg.q.to(dev), xg.k.to(dev), xg.v.to(dev), causal=True, scale=xg.scale)
            xv = inputs.varlen_config()
            fattn.fwd(xv.q.to(dev), xv.k.to(dev), xv.v.to(dev), causal=True, scale=xv.scale,
                      cu_seqlens=xv.cu_seqlens.to(dev), max_seqlen=xv.max_seqlen)
        torch.cuda.synchronize()
        st = fattn.debug_read_status()
        print(json.dumps({"profile_once": True, "num_splits": S, "device_status": st}), flush=True)
        if st != 0:
            raise SystemExit(1)
        return

    for _ in range(max(3, args.warmup)):
        flush()
        prefill()
        flush()
        decode()
    torch.cuda.synchronize()
    assert fattn.debug_read_status() == 0

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for s in range(args.steps):
        flush()
        ev[s][0].record(stream)
        prefill()
        ev[s][1].record(stream)
        flush()
        ev[s][2].record(stream)
        decode()
        ev[s][3].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t_wall = time.perf_counter() - t_wall
    clocks = sampler.stop()
    launches = 2 * args.steps  # per step: prefill_tc_kernel, decode_kernel (+ the counter memset, a driver op)
    status = fattn.debug_read_status()

    pre_ms = [e[0].elapsed_time(e[1]) for e in ev]
    dec_ms = [e[2].elapsed_time(e[3]) for e in ev]
    t_pre = sum(pre_ms) / len(pre_ms)
    t_dec = sum(dec_ms) / len(dec_ms)
    t_pre, t_dec = max_over_ranks([t_pre, t_dec], world, dev)

    flops = pre.flops()
    kv_bytes = dec.kv_bytes()
    tflops = flops / (t_pre * 1e-3) / 1e12
    gbs = kv_bytes / (t_dec * 1e-3) / 1e9
    peaks, peak_src = load_peaks()

    # ---------------------------------------------------------------- e2e through host buffers
    e2e = None
    if not args.no_e2e:
        hq_, hk_, hv_ = pre.q.pin_memory(), pre.k.pin_memory(), pre.v.pin_memory()
        ho = torch.empty_like(pre.q).pin_memory()
        hl = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        hdq, hdk, hdv = dec.q.pin_memory(), dec.kcache.pin_memory(), dec.vcache.pin_memory()
        hbt, hsl = dec.block_table.pin_memory(), dec.seqlens.pin_memory()
        hdo = torch.empty_like(dec.q).pin_memory()
        hdl = torch.empty((dec.batch, dec.hq), dtype=torch.float32).pin_memory()
        h2d_pre = sum(t.numel() * t.element_size() for t in (hq_, hk_, hv_))
        d2h_pre = ho.numel() * ho.element_size() + hl.numel() * 4
        h2d_dec = sum(t.numel() * t.element_size() for t in (hdq, hdk, hdv, hbt, hsl))
        d2h_dec = hdo.numel() * hdo.element_size() + hdl.numel() * 4

        # Double-buffered pipeline on three streams: step k's inputs are copied in while step
        # k-1 computes and step k-2's outputs are copied out; a buffer set is refilled only
        # after the kernel that read it finished, and a kernel writes an output set only
        # after that set's previous copy-out finished. Every step's copies and kernel lie
        # inside the timed region (first copy-in to last copy-out, fill and drain included).
        s_in, s_cmp, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

        def pipelined(n, h_in, d_in, run, d_out, h_out):
            ev_in, ev_cmp, ev_out = ([torch.cuda.Event() for _ in range(n)] for _ in range(3))
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            main = torch.cuda.current_stream()
            t0.record(main)
            for st in (s_in, s_cmp, s_out):
                st.wait_event(t0)
            for i in range(n):
                b = i % 2
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(ev_cmp[i - 2])
                    for dt, ht in zip(d_in[b], h_in):
                        dt.copy_(ht, non_blocking=True)
                    ev_in[i].record(s_in)
                with torch.cuda.stream(s_cmp):
                    s_cmp.wait_event(ev_in[i])
                    if i >= 2:
                        s_cmp.wait_event(ev_out[i - 2])
                    run(b)
                    ev_cmp[i].record(s_cmp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_cmp[i])
                    for ht, dt in zip(h_out[b], d_out[b]):
                        ht.copy_(dt, non_blocking=True)
                    ev_out[i].record(s_out)
            main.wait_event(ev_out[n - 1])
            t1.record(main)
            torch.cuda.synchronize()
            return t0.elapsed_time(t1) / n

        pre_in = [(q, k, v), (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))]
        pre_out = [(o, lse), (torch.empty_like(o), torch.empty_like(lse))]
        pre_hout = [(ho, hl), (torch.empty_like(ho).pin_memory(), torch.empty_like(hl).pin_memory())]

        def run_pre(b):
            (qq, kk, vv), (oo, ll) = pre_in[b], pre_out[b]
            fattn.fwd(qq, kk, vv, causal=True, scale=pre.scale, out=oo, lse=ll)

        dec_in = [(dq, dk, dv, dbt, dsl), tuple(torch.empty_like(t) for t in (dq, dk, dv, dbt, dsl))]
        dec_out = [(do, dlse), (torch.empty_like(do), torch.empty_like(dlse))]
        dec_hout = [(hdo, hdl), (torch.empty_like(hdo).pin_memory(), torch.empty_like(hdl).pin_memory())]

        def run_dec(b):
            (a, kc, vc, bt, sl), (oo, ll) = dec_in[b], dec_out[b]
            fattn.decode_paged(a, kc, vc, bt, sl, S, scale=dec.scale, out=oo, lse=ll, workspace=ws)

        n_e2e = max(4, min(args.steps, 10))
        pipelined(2, (hq_, hk_, hv_), pre_in, run_pre, pre_out, pre_hout)  # warm-up
        pipelined(2, (hdq, hdk, hdv, hbt, hsl), dec_in, run_dec, dec_out, dec_hout)
        tp = pipelined(n_e2e, (hq_, hk_, hv_), pre_in, run_pre, pre_out, pre_hout)
        td = pipelined(n_e2e, (hdq, hdk, hdv, hbt, hsl), dec_in, run_dec, dec_out, dec_hout)
        tp, td = max_over_ranks([tp, td], world, dev)
        e2e = {"value": world * flops / (tp * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d_pre + h2d_dec, "d2h_bytes_per_step": d2h_pre + d2h_dec,
               "prefill_ms": tp, "decode_ms": td, "steps": n_e2e,
               "overlap": "double-buffered, three streams: step k+1's host-to-device copy runs during "
                          "step k's kernel and device-to-host copy",
               "decode": {"value": world * kv_bytes / (td * 1e-3) / 1e9, "unit": "GB/s"}}

    sparse = None if args.no_sparse else block_sparse_leg(fattn, pre, q, k, v, o, lse, flush, stream, peaks)
    paged = None if args.no_sparse else paged_prefill_leg(fattn, flush, stream, peaks, dev)
    backward = None if args.no_sparse else backward_leg(fattn, pre, q, k, v, o, lse, flush, stream, peaks, dev)
    masked = None if args.no_sparse else masked_leg(fattn, pre, q, k, v, o, lse, flush, stream, peaks, dev)
    fp8 = None if args.no_sparse else fp8_leg(fattn, pre, flush, stream, peaks, dev)
    cpu_s = 0.0 if (rank != 0 or world != 1 or args.no_cpu_baseline) else args.cpu_leg_seconds
    from exact_tiled_attention_fattn_gb300 import inputs as _inputs
    long_gqa = None if args.no_configs else prefill_config_leg(
        fattn, _inputs.long_gqa_config(), "long-context GQA causal prefill B=1 Hq=32 Hkv=8 N=32768 d=128 (seed 2)",
        "prefill_tc_kernel<128>, long GQA", flush, stream, peaks, dev, cpu_s)
    varlen = None if args.no_configs else prefill_config_leg(
        fattn, _inputs.varlen_config(), "ragged varlen causal prefill, 16 sequences U[128,2048] (seed 3, T=13794) "
        "Hq=Hkv=16 d=64", "prefill_tc_kernel<64>, varlen", flush, stream, peaks, dev, cpu_s)

    cpu = cpu_dec = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_prefill(pre, args.cpu_seconds)
        cpu_dec = cpu_baseline_decode(dec, args.cpu_leg_seconds)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    peak_t = peaks["bf16_tflops"]
    peak_b = peaks["hbm_gbs"]
    line = {
        "metric": METRIC,
        "value": world * tflops,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t_pre + t_dec,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "causal MHA prefill B=4 Hq=Hkv=32 N=4096 d=128 + paged split-KV decode "
                               "B=8 Hq=32 Hkv=8 d=128 ctx U[1024,65536] seed 4, 16-token pages",
                   "parallelism": f"replicas x{world}", "num_splits": S,
                   "l2": "flushed before every timed launch: 256 MB written, then a separate 256 MB read"},
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak_t, "unit": "TFLOP/s",
                     "frac": tflops / peak_t, "traffic": recorded_traffic("prefill_tc_kernel<128>"),
                     "peak_source": f"{peak_src} bf16_tflops (burst)", "kernel": "prefill_tc_kernel<128>"},
        "decode": {"value": world * gbs, "unit": "GB/s", "ms": t_dec, "kv_bytes": kv_bytes,
                   "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak_b, "unit": "GB/s",
                                "frac": gbs / peak_b, "traffic": recorded_traffic("decode_kernel<128, page16>"),
                                "peak_source": f"{peak_src} hbm_gbs", "kernel": "decode_kernel<128, page16>"},
                   "cpu_baseline": cpu_dec},
        "prefill_ms": t_pre,
        "long_gqa_prefill": long_gqa,
        "varlen_prefill": varlen,
        "block_sparse": sparse,
        "paged_prefill": paged,
        "backward": backward,
        "masked_prefill": masked,
        "fp8_prefill": fp8,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "gpu_launches": launches,
        "device_status": status,
        "wall_s_timed": t_wall,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
