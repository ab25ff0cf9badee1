#!/usr/bin/env python
"""Throughput of the exact-attention hot path on GB300 (one JSON line on stdout).

A step is one pass of the whole path over one batch: the tensor-core forward (O, lse) and, for
workloads with a backward, the recomputing backward (dQ, dK, dV) -- every launch goes through the
C ABI of libfa_gb300.so. The default workload is the long-sequence causal forward B=8, H=32,
N=8192, d=128, bf16 (the largest specified problem); the same line carries a `per_config` object
with one entry for each of the other specified workloads (the fp32 single head, the multi-head
N=2048 forward, the block-sparse N=16384 forward and the causal N=4096 backward), each timed
the same way, with its own roofline fraction, clocks and oracle baseline, and a `next_rows` object
with the FP8 (e4m3) forward on the long-sequence shape, measured against the fp8 peak, the bf16
forwards of the long-sequence and multi-head workloads with part of the exponentials computed in
software (fa_set_exp2_emulation), which is off by default, and decoding with eight query rows per
head against a 32768-key cache, in GB/s against the measured copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--backward]
                  [--no-per-config] [--impl ours|reference]

Metric: TFLOPS = algorithmic FLOPs / time, with 4*B*H*N^2*d for the forward (causal: half;
block-sparse: active tiles only) and 2.5 times that for the backward (its five contractions).
`value` is timed with CUDA events around the kernels only (inputs resident in HBM, L2 flushed
between steps outside the events by writing a 512 MiB buffer and reading half of it back, so that
no dirty line of the flush is left to be written back during the timed kernels); `e2e` is the
same step through the public API from pinned host buffers, host<->device copies inside the timed
region (no flush there: every step's inputs arrive fresh from the host). Under torchrun every
rank runs its own replica of the workload (independent heads: no collective on the data path)
and `value` sums over ranks using the slowest rank's time.

Decoding workloads (decode_*: a few query rows per head against a long key/value cache) are
bound by HBM bandwidth, so their line reports GB/s of algorithmic bytes (K and V read once, q
read, O and lse written) against the measured copy bandwidth.

--impl reference times the fp64 CPU oracle (the parity reference) on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "causal_N8192_d128"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Datasheet figures for one GB300 (dense, no sparsity), reported beside the measured peaks.
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 7900.0
FP8_OVER_BF16 = 4.5 / 2.25  # datasheet dense fp8 / bf16 tensor rates
FP32_FMA_PER_CLK_PER_SM = 128  # fp32 FMA lanes per SM (four sub-partitions of 32)
FLUSH_BYTES = 512 << 20        # > the 129 MB L2
# Oracle rows per CPU task for forward-only workloads (a strided subset of one head's query rows).
ORACLE_ROWS_PER_TASK = 256
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--backward", action="store_true",
                    help="add the backward to a forward workload's step")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-configuration entries of the default line")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args(argv)


def bench_workload(name: str, backward: bool = False):
    from exact_attention_fa_gb300 import workloads as wl
    w = wl.WORKLOADS[name]
    return w.with_(backward=True) if backward and not w.decode else w


def per_config_names(main_name: str):
    """The specified workloads other than the line's own, in their specified order."""
    from exact_attention_fa_gb300 import workloads as wl
    return [n for n in wl.SPECIFIED if n != main_name]


# Workloads of rows past the specified ones, measured beside them on the default line: the FP8
# forward on the long-sequence causal shape.
NEXT_ROWS = ["causal_N8192_d128_fp8"]
# ... and decoding (split keys + merge) with eight new query rows per head, in GB/s against HBM.
NEXT_DECODE = "decode_N32768_d128_q8_b2"
EXP2_EMULATION_PER32 = 4  # fa_set_exp2_emulation's setting measured on the default line


def flops(w, mask=None):
    from exact_attention_fa_gb300 import workloads as wl
    f = wl.flop_count(w, mask, "fwd")
    return f, (2.5 * f if w.backward else 0.0)


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def metric_name(w):
    if w.decode:
        return "attention decode GB/s (K, V read once; q, O, lse)"
    return "attention fwd/bwd TFLOPS (4·B·H·N²·d, causal halved)"


def unit_of(w):
    return "GB/s" if w.decode else "TFLOPS"


def config_of(w, n_gpus, note=None):
    c = {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "dtype": w.dtype,
         **({"Nq": w.nq, "Nk": w.N} if w.decode else {}),
         "causal": w.causal, "block_sparse": w.block_sparse,
         "step": "forward+backward" if w.backward else "forward",
         "global_batch": w.B * n_gpus, "seq_len": w.N, "parallelism": f"replicas{n_gpus}",
         "l2": "flushed between timed steps outside the timed events (512 MiB write, "
               "then 256 MiB of it read back: no input and no dirty line left in L2)"}
    if note:
        c["note"] = note
    return c


# ----------------------------------------------------------------------------------------- CPU
# The oracle as it stands, timed on a bounded sample of the workload: tasks of whole heads
# (backward, decoding) or of a strided subset of one head's query rows (forward; rows are
# independent, so the subset is the same computation restricted to those rows).

def row_stride(w) -> int:
    if w.backward or w.decode:
        return 1
    return max(1, w.N // ORACLE_ROWS_PER_TASK)


def oracle_tasks(w, inp, first, count):
    """Tasks first .. first+count-1: task i takes head i mod B*H and, for forward workloads, the
    query rows offset, offset + stride, ... with offset = (i div B*H) mod stride, so consecutive
    rounds walk every head before they repeat one. Returns (tasks, work in the metric's unit)."""
    import numpy as np
    from exact_attention_fa_gb300 import workloads as wl
    mask = inp.raw("mask") if w.block_sparse else None
    BH = w.B * w.H
    stride = row_stride(w)
    if w.decode:
        per_head = wl.decode_bytes(w) / BH / 1e9
        tile_work = None
    else:
        f_fwd, f_bwd = flops(w, mask)
        per_head = (f_fwd + f_bwd) / BH / 1e12
        # block-sparse: the metric's work of one query row is 4 d 128 per active tile of its row
        tile_work = (4.0 * w.d * wl.TILE * mask.sum(axis=1) / 1e12
                     if w.block_sparse and not w.causal else None)
    tasks, work = [], 0.0
    for i in range(first, first + count):
        b, h = divmod(i % BH, w.H)
        rows = None
        if stride > 1:
            rows = np.arange((i // BH) % stride, w.N, stride)
        do = inp.raw("do")[b, h] if w.backward else None
        tasks.append((inp.raw("q")[b, h], inp.raw("k")[b, h], inp.raw("v")[b, h], do,
                      w.softmax_scale, w.causal, mask, rows))
        if rows is None:
            work += per_head
        elif tile_work is not None:
            work += float(tile_work[rows // wl.TILE].sum())
        else:
            work += per_head * rows.size / w.N
    return tasks, work


def make_pool(cores):
    import multiprocessing as mp
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"  # one BLAS thread per worker: `cores` threads in total
    from oracle import cpu_baseline
    pool = mp.get_context("spawn").Pool(cores)
    pool.map(cpu_baseline.warm, range(cores))
    return pool


def time_oracle(pool, tasks):
    from oracle import cpu_baseline
    t0 = time.perf_counter()
    pool.map(cpu_baseline.run_head, tasks, chunksize=1)
    return time.perf_counter() - t0


def describe_sample(w, n_tasks):
    BH = w.B * w.H
    stride = row_stride(w)
    part = "forward+backward" if w.backward else "forward"
    if stride > 1:
        what = (f"{n_tasks} tasks of {len(range(0, w.N, stride))} query rows (every "
                f"{stride}th row of one head; {min(n_tasks, BH)} of {BH} heads)")
    else:
        what = f"{n_tasks} whole heads ({min(n_tasks, BH)} distinct of {BH})"
    return f"{what} of {w.name}, fp64 numpy oracle ({part}), one task per worker"


def cpu_baseline_leg(pool, cores, w, inp, budget_s=20.0, min_s=2.0):
    """The oracle on a bounded sample of the workload, on all host cores: rounds of `cores` tasks
    until the budget is spent, or every head was visited and at least min_s has passed."""
    BH = w.B * w.H
    done, total, work = 0, 0.0, 0.0
    while True:
        tasks, wk = oracle_tasks(w, inp, done, cores)
        dt = time_oracle(pool, tasks)
        done += len(tasks)
        total += dt
        work += wk
        if total + dt > budget_s or (done >= BH and total >= min_s):
            break
    return {"value": work / total, "unit": unit_of(w), "cores": cores, "kind": "oracle",
            "sample": describe_sample(w, done), "seconds": round(total, 3)}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = bench_workload(args.workload, args.backward)
    from exact_attention_fa_gb300 import workloads as wl
    inp = wl.make_inputs(w, with_do=w.backward)
    cores = host_cores()
    pool = make_pool(cores)
    times, works = [], []
    try:
        for i in range(args.warmup + args.steps):
            tasks, wk = oracle_tasks(w, inp, i * cores, cores)
            dt = time_oracle(pool, tasks)
            if i >= args.warmup:
                times.append(dt)
                works.append(wk)
    finally:
        pool.terminate()
    t = statistics.fmean(times)
    value = sum(works) / sum(times)
    print(json.dumps({
        "impl": "reference", "metric": metric_name(w), "value": value, "unit": unit_of(w),
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args.gpus),
        "cpu_baseline": {"value": value, "unit": unit_of(w), "cores": cores, "kind": "oracle",
                         "sample": "per step: " + describe_sample(w, cores)},
        "e2e": {"value": value, "unit": unit_of(w), "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


# ----------------------------------------------------------------------------------------- GPU

def aggregate_over_ranks(local_ms, world, device=None):
    """Each timing's maximum over ranks: the slowest replica sets the job's time."""
    if world == 1:
        return list(local_ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(local_ms), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_tflops(world, flops_per_rank, ms):
    """Whole-job throughput: every replica processes flops_per_rank in the job time ms."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def fp32_peak_tflops(peaks) -> float:
    """fp32 FMA peak from unit counts and clock: SMs x 128 FMA/clk x 2 FLOP x max SM clock."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    mhz = float(peaks.get("sm_max_mhz", 2070.0))
    return sms * FP32_FMA_PER_CLK_PER_SM * 2 * mhz * 1e6 / 1e12


class ClockSampler:
    """nvidia-smi's clocks and throttle reasons sampled every 50 ms while the block runs
    (read-only queries)."""

    def __init__(self, path):
        self.path = path
        self.proc = None

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self, device_index):
        if self.proc is None:
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9 or parts[0] != str(device_index):
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def forward_kernel_name(w):
    """Name of the forward kernel the library runs for this workload (the two-query-tile kernel
    for every bf16 and e4m3 forward). fp32: small problems at d <= 96 (8-row CTAs would leave SMs
    idle, and a CTA's whole key range fits in 200 KB of shared memory) take the kernel that stages
    all keys at once; the rest the key-block kernel."""
    if w.dtype == "fp32":
        import torch
        sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
        smem = 4 * (w.N * (w.d + 4) + w.N * w.d + 2 * w.d + 16 * (w.d + 2))
        if (w.N + 7) // 8 * w.B * w.H < sms and w.d <= 96 and smem <= 200 * 1024:
            return f"fwd_fp32_small_kernel<{w.d}>"
        return f"fwd_fp32_kernel<{w.d}>"
    if w.dtype == "e4m3":
        return f"fwd_pair_kernel<{w.d}, true>"
    return f"fwd_pair_kernel<{w.d}>"


def recorded_traffic(kname, w):
    """DRAM bytes per launch of the dominant kernel from a committed ncu summary, if one exists
    for this kernel, workload and kernel source; otherwise None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    from exact_attention_fa_gb300 import build
    entry = rec.get(f"{w.name}:{kname.split(' (')[0]}")
    if not entry or entry.get("source_digest") != build.source_digest():
        return None
    return entry.get("dram_bytes_per_launch")


class Problem:
    """One attention workload's device tensors and its forward / backward calls (C ABI)."""

    def __init__(self, w, inp, fa, dev):
        import numpy as np
        import torch
        self.w, self.fa = w, fa

        def dev_tensor(name):
            a = inp.raw(name)
            if a.dtype == np.uint16:
                return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
            if a.dtype == np.uint8 and name != "mask":  # e4m3 codes
                return torch.from_numpy(a).to(dev).view(torch.float8_e4m3fn)
            return torch.from_numpy(a).to(dev)

        self.q, self.k, self.v = dev_tensor("q"), dev_tensor("k"), dev_tensor("v")
        self.do = dev_tensor("do") if w.backward else None
        self.mask = dev_tensor("mask") if w.block_sparse else None
        self.o = (torch.empty(self.q.shape, dtype=torch.bfloat16, device=dev)
                  if w.dtype == "e4m3" else torch.empty_like(self.q))
        self.lse = torch.empty(self.q.shape[:3], dtype=torch.float32, device=dev)
        if w.backward:
            self.dq = torch.empty(self.q.shape, dtype=torch.float32, device=dev)
            self.dk, self.dv = torch.empty_like(self.k), torch.empty_like(self.v)
            self.ws = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.N, w.d),
                                  dtype=torch.uint8, device=dev)
        self.f_fwd, self.f_bwd = flops(w, inp.raw("mask") if w.block_sparse else None)
        self.launches = 1 + (2 if w.backward else 0)

    def fwd(self, q=None, k=None, v=None, o=None, lse=None):
        w, fa = self.w, self.fa
        q, k, v = (self.q if q is None else q), (self.k if k is None else k), (self.v if v is None else v)
        o, lse = (self.o if o is None else o), (self.lse if lse is None else lse)
        if w.dtype == "fp32":
            fa.fa_fwd_fp32(q, k, v, o, lse, w.softmax_scale, w.causal)
        elif w.dtype == "e4m3":
            fa.fa_fwd_fp8(q, k, v, o, lse, w.softmax_scale, 1.0, w.causal)
        elif w.block_sparse:
            fa.fa_fwd_blocksparse(q, k, v, o, lse, w.softmax_scale, self.mask, w.causal)
        else:
            fa.fa_fwd(q, k, v, o, lse, w.softmax_scale, w.causal)

    def bwd(self, q=None, k=None, v=None, o=None, do=None, lse=None, dq=None, dk=None, dv=None,
            ws=None):
        pick = lambda a, b: b if a is None else a  # noqa: E731
        w = self.w
        self.fa.fa_bwd(pick(q, self.q), pick(k, self.k), pick(v, self.v), pick(o, self.o),
                       pick(do, self.do), pick(lse, self.lse), pick(dq, self.dq),
                       pick(dk, self.dk), pick(dv, self.dv), w.softmax_scale, w.causal,
                       pick(ws, self.ws))

    def dominant(self, t_fwd, t_bwd):
        """(kernel name, FLOPs, ms) of the part of the step that takes longer."""
        w = self.w
        if w.backward and t_bwd >= t_fwd:
            return (f"bwd_tc_kernel<{w.d}> (+ bwd_prep_kernel<{w.d}> in the same call)",
                    self.f_bwd, t_bwd)
        return forward_kernel_name(w), self.f_fwd, t_fwd


def flush_l2(buf):
    """Evicts every input from L2 before a timed step: writes the whole buffer (larger than L2),
    then reads its first half back, so that L2 ends up holding clean lines of this buffer only and
    the timed kernels pay for none of the flush's dirty lines being written back."""
    import torch
    buf.zero_()
    buf[: buf.numel() // 2].view(torch.int64).sum()


def time_problem(pr, steps, warmup, flush_buf, world, dev, local):
    """CUDA-event times (ms, averaged over `steps`, max over ranks) of the forward, the backward
    and the whole step, with L2 flushed before every step outside the events; nvidia-smi clocks
    are sampled during the timed region."""
    import torch
    import torch.distributed as dist
    for _ in range(warmup):
        flush_l2(flush_buf)
        pr.fwd()
        if pr.w.backward:
            pr.bwd()
    pr.fa.fa_check_device_error(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(os.path.join("/tmp", f"fa_clocks_{os.getpid()}.csv")) as clocks:
        time.sleep(0.1)
        t0 = time.perf_counter()
        for i in range(steps):
            flush_l2(flush_buf)
            ev[i][0].record()
            pr.fwd()
            ev[i][1].record()
            if pr.w.backward:
                pr.bwd()
            ev[i][2].record()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        wall = time.perf_counter() - t0
        time.sleep(0.1)
    pr.fa.fa_check_device_error(dev)
    step_ms = statistics.fmean(ev[i][0].elapsed_time(ev[i][2]) for i in range(steps))
    fwd_ms = statistics.fmean(ev[i][0].elapsed_time(ev[i][1]) for i in range(steps))
    bwd_ms = (statistics.fmean(ev[i][1].elapsed_time(ev[i][2]) for i in range(steps))
              if pr.w.backward else 0.0)
    per_step = [ev[i][0].elapsed_time(ev[i][2]) for i in range(steps)]
    med_ms, min_ms = statistics.median(per_step), min(per_step)
    step_ms, fwd_ms, bwd_ms, med_ms, min_ms = aggregate_over_ranks(
        [step_ms, fwd_ms, bwd_ms, med_ms, min_ms], world, dev)
    return {"step_ms": step_ms, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "step_ms_median": med_ms,
            "step_ms_min": min_ms, "clocks": clocks.summary(local), "wall_s": wall}


def roofline_of(pr, kname, kflops, kms, peaks, peak_src):
    """The dominant kernel against its roofline: the tensor pipe's measured bf16 peak, or for the
    fp32 path the FMA pipes' peak derived from unit counts and the clock."""
    achieved = kflops / (kms * 1e-3) / 1e12
    traffic = recorded_traffic(kname, pr.w)
    if pr.w.dtype == "fp32":
        alu_peak = fp32_peak_tflops(peaks)
        return {"bound": "alu", "kernel": kname, "achieved": achieved, "peak": alu_peak,
                "unit": "TFLOP/s", "frac": achieved / alu_peak,
                "peak_source": "derived: SMs x 128 fp32 FMA/clk x 2 x max SM clock",
                "traffic": traffic}
    peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    src = "MEASURED_PEAKS.json" if peak_src == "measured" else "fallback"
    nominal, what = NOMINAL_BF16_TFLOPS, f"{peak_src} bf16 dense (burst) {src}"
    if pr.w.dtype == "e4m3":
        # an fp8 contraction: the measured bf16 peak times the datasheet fp8 / bf16 ratio (2)
        peak, sustained, nominal = (FP8_OVER_BF16 * x for x in (peak, sustained, nominal))
        what = f"{peak_src} bf16 dense (burst) {src} x {FP8_OVER_BF16:g} (datasheet fp8 / bf16)"
    return {"bound": "tensor", "kernel": kname, "achieved": achieved, "peak": peak,
            "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": what,
            "frac_of_sustained": achieved / sustained,
            "frac_of_nominal": achieved / nominal, "nominal": nominal,
            "traffic": traffic}


def parts_of(pr, t, peak):
    out = {"fwd": {"ms": t["fwd_ms"], "tflops": pr.f_fwd / (t["fwd_ms"] * 1e-3) / 1e12}}
    out["fwd"]["frac_of_bf16_peak"] = out["fwd"]["tflops"] / peak
    if pr.w.backward:
        tf = pr.f_bwd / (t["bwd_ms"] * 1e-3) / 1e12
        # the backward counts its five contractions (2.5x the forward's FLOP); the metric's
        # literal 4*B*H*N^2*d (causal halved) over the backward's time is reported beside it
        out["bwd"] = {"ms": t["bwd_ms"], "tflops": tf, "frac_of_bf16_peak": tf / peak,
                      "tflops_at_literal_4BHN2d": pr.f_fwd / (t["bwd_ms"] * 1e-3) / 1e12}
    return out


def e2e_leg(pr, steps, world, dev):
    """The step end to end through the public API from pinned host buffers: each step copies its
    inputs (Q, K, V and, with the backward, dO) host->device, runs the step, and reads every result
    back (O, lse and dQ, dK, dV). Steps are pipelined the way a training loop prefetches: two sets
    of device buffers; the host->device copy of step i+1 and the device->host copy of step i-1 run
    on their own streams while step i computes."""
    import torch
    w = pr.w
    host_in = {n: t.cpu().pin_memory() for n, t in (("q", pr.q), ("k", pr.k), ("v", pr.v))}
    if w.backward:
        host_in["do"] = pr.do.cpu().pin_memory()
    out_names = ["o", "lse"] + (["dq", "dk", "dv"] if w.backward else [])
    proto = {"o": pr.o, "lse": pr.lse}
    if w.backward:
        proto.update(dq=pr.dq, dk=pr.dk, dv=pr.dv)
    sets = []
    for _ in range(2):
        dev_in = {n: torch.empty_like(t, device=dev) for n, t in host_in.items()}
        dev_out = {n: torch.empty_like(proto[n]) for n in out_names}
        host_out = {n: torch.empty(proto[n].shape, dtype=proto[n].dtype, pin_memory=True)
                    for n in out_names}
        ws = torch.empty_like(pr.ws) if w.backward else None
        sets.append((dev_in, dev_out, host_out, ws))
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in sets[0][2].values())
    s_comp, s_h2d, s_d2h = (torch.cuda.Stream(dev) for _ in range(3))

    def step(b):
        di, do_, _, ws = sets[b]
        pr.fwd(di["q"], di["k"], di["v"], do_["o"], do_["lse"])
        if w.backward:
            pr.bwd(di["q"], di["k"], di["v"], do_["o"], di["do"], do_["lse"], do_["dq"],
                   do_["dk"], do_["dv"], ws)

    E = max(1, min(steps, 100))
    W2 = 2  # untimed pipelined steps first
    n_tot = W2 + E
    ev_in = [torch.cuda.Event() for _ in range(n_tot)]
    ev_comp = [torch.cuda.Event() for _ in range(n_tot)]
    ev_out = [torch.cuda.Event() for _ in range(n_tot)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    for i in range(n_tot):
        b = i % 2
        di, do_, ho, _ = sets[b]
        if i == W2:
            torch.cuda.synchronize()
            t_start.record(s_h2d)
            s_comp.wait_event(t_start)
            s_d2h.wait_event(t_start)
        with torch.cuda.stream(s_h2d):
            if i >= 2:
                s_h2d.wait_event(ev_comp[i - 2])  # buffer set b no longer read by step i-2
            for n, t in host_in.items():
                di[n].copy_(t, non_blocking=True)
            ev_in[i].record(s_h2d)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev_in[i])
            if i >= 2:
                s_comp.wait_event(ev_out[i - 2])  # outputs of step i-2 were read back
            step(b)
            ev_comp[i].record(s_comp)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(ev_comp[i])
            for n in out_names:
                ho[n].copy_(do_[n], non_blocking=True)
            ev_out[i].record(s_d2h)
    s_d2h.wait_event(ev_out[n_tot - 1])
    t_end.record(s_d2h)
    torch.cuda.synchronize()
    pr.fa.fa_check_device_error(dev)
    t_e2e = aggregate_over_ranks([t_start.elapsed_time(t_end) / E], world, dev)[0]
    return {"value": job_tflops(world, pr.f_fwd + pr.f_bwd, t_e2e), "unit": "TFLOPS",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e,
            "steps": E, "pipelined": "host->device, compute and device->host of consecutive "
                                     "steps overlap on three streams (two buffer sets)",
            "l2": "not flushed: every step's inputs are copied in from the host"}


def per_config_steps(t_est_ms, steps):
    """Steps for a per-configuration entry: at least `steps` (capped at 100) and enough for the
    timed region to last about half a second, so the clock sampler sees it; at most 2000."""
    want = math.ceil(500.0 / max(t_est_ms, 1e-3))
    return int(max(min(steps, 100), min(want, 2000)))


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = bench_workload(args.workload, args.backward)
    from exact_attention_fa_gb300 import workloads as wl
    default_line = not args.no_per_config and not w.decode and args.workload == DEFAULT_WORKLOAD
    others = per_config_names(w.name) if default_line else []
    nexts = list(NEXT_ROWS) if default_line else []
    cfg_w = {n: wl.WORKLOADS[n] for n in others + nexts}
    dec_w = wl.WORKLOADS[NEXT_DECODE] if default_line else None

    # host inputs first; the oracle's worker pool (spawned) runs before CUDA is touched
    inp = wl.make_inputs(w, with_do=w.backward)
    cfg_inp = {n: wl.make_inputs(cw, with_do=cw.backward) for n, cw in cfg_w.items()}
    dec_inp = wl.make_inputs(dec_w) if dec_w is not None else None
    cpu, cfg_cpu = None, {}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = host_cores()
        pool = make_pool(cores)
        try:
            cpu = cpu_baseline_leg(pool, cores, w, inp, budget_s=20.0, min_s=10.0)
            for n, cw in cfg_w.items():
                cfg_cpu[n] = cpu_baseline_leg(pool, cores, cw, cfg_inp[n], budget_s=6.0)
            if dec_w is not None:
                cfg_cpu[NEXT_DECODE] = cpu_baseline_leg(pool, cores, dec_w, dec_inp, budget_s=6.0)
        finally:
            pool.terminate()

    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import exact_attention_fa_gb300 as fa
    fa.load()
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    if w.decode:
        return run_decode(args, w, fa, inp, cpu, world, rank, local, dev, flush_buf)

    pr = Problem(w, inp, fa, dev)
    K = args.steps
    t = time_problem(pr, K, args.warmup, flush_buf, world, dev, local)
    e2e = None if args.no_e2e else e2e_leg(pr, K, world, dev)

    peaks, peak_src = load_peaks()
    peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])

    def measure(cpr, n):
        # a short probe sets the step count, then the timed run
        probe = time_problem(cpr, 3, max(3, min(args.warmup, 5)), flush_buf, world, dev, local)
        steps = per_config_steps(probe["step_ms"], K)
        ct = time_problem(cpr, steps, max(3, args.warmup), flush_buf, world, dev, local)
        kname, kflops, kms = cpr.dominant(ct["fwd_ms"], ct["bwd_ms"])
        return {
            "config": config_of(cpr.w, world),
            "ms_per_step": ct["step_ms"], "steps": steps,
            "tflops": job_tflops(world, cpr.f_fwd + cpr.f_bwd, ct["step_ms"]),
            "parts": parts_of(cpr, ct, peak),
            "roofline": roofline_of(cpr, kname, kflops, kms, peaks, peak_src),
            "cpu_baseline": cfg_cpu.get(n),
            "gpu_launches": cpr.launches * steps,
            "clocks": ct["clocks"],
        }

    per_config, next_rows = {}, {}
    for n, cw in cfg_w.items():
        cpr = Problem(cw, cfg_inp[n], fa, dev)
        (next_rows if n in nexts else per_config)[n] = measure(cpr, n)
        del cpr
    if default_line:
        # the partial software exponential (4 of every 32 exponentials per row on the FMA
        # pipes), off by default, measured beside the default on the same problems
        for n, cpr in ((w.name, pr),
                       ("mha_N2048_d64", Problem(cfg_w["mha_N2048_d64"],
                                                 cfg_inp["mha_N2048_d64"], fa, dev))):
            fa.fa_set_exp2_emulation(EXP2_EMULATION_PER32)
            try:
                e = measure(cpr, n)
            finally:
                fa.fa_set_exp2_emulation(0)
            e["exp2_emulation_per32"] = EXP2_EMULATION_PER32
            e["roofline"]["kernel"] += f" ({EXP2_EMULATION_PER32} of 32 exponentials in software)"
            e["roofline"]["traffic"] = None  # the traffic record is the default instance's
            next_rows[f"{n}+exp2_emulation"] = e
        next_rows[NEXT_DECODE] = decode_entry(dec_w, dec_inp, fa, dev, flush_buf, K,
                                              max(3, args.warmup), world, local,
                                              cfg_cpu.get(NEXT_DECODE))

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    kname, kflops, kms = pr.dominant(t["fwd_ms"], t["bwd_ms"])
    line = {
        "metric": metric_name(w), "value": job_tflops(world, pr.f_fwd + pr.f_bwd, t["step_ms"]),
        "unit": "TFLOPS", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": t["step_ms"], "higher_is_better": True, "scaling": "weak",
        "ms_per_step_median": t["step_ms_median"], "ms_per_step_min": t["step_ms_min"],
        "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic: i.i.d. N(0,1) inputs, seeded"
                + {"bf16": ", rounded to bf16", "e4m3": ", rounded to e4m3"}.get(w.dtype, ""),
        "config": config_of(w, world),
        "parts": parts_of(pr, t, peak),
        "roofline": roofline_of(pr, kname, kflops, kms, peaks, peak_src),
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": pr.launches * K,
        "clocks": t["clocks"],
        "wall_s_timed_region": t["wall_s"],
    }
    if per_config:
        line["per_config"] = per_config
    if next_rows:
        line["next_rows"] = next_rows
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def decode_entry(w, inp, fa, dev, flush_buf, steps, warmup, world, local, cpu=None):
    """A decoding workload timed like the per-configuration entries (CUDA events around each
    fa_decode call, L2 flushed before each, clocks sampled), reported in GB/s of algorithmic bytes
    against the measured copy bandwidth."""
    import numpy as np
    import torch
    import torch.distributed as dist
    from exact_attention_fa_gb300 import workloads as wl

    def dev_tensor(name):
        return torch.from_numpy(inp.raw(name).view(np.int16)).to(dev).view(torch.bfloat16)

    q, k, v = dev_tensor("q"), dev_tensor("k"), dev_tensor("v")
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    n_ctas = fa.fa_decode_ctas(w.B, w.H, w.nq, w.N, w.d)
    ws = torch.empty(fa.fa_decode_workspace_bytes(w.B, w.H, w.nq, w.N, w.d), dtype=torch.uint8,
                     device=dev)
    algo_bytes = wl.decode_bytes(w)

    def timed(n):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        for i in range(n):
            flush_l2(flush_buf)
            ev[i][0].record()
            fa.fa_decode(q, k, v, o, lse, w.softmax_scale, n_ctas, ws)
            ev[i][1].record()
        torch.cuda.synchronize()
        return statistics.fmean(ev[i][0].elapsed_time(ev[i][1]) for i in range(n))

    for _ in range(warmup):
        flush_l2(flush_buf)
        fa.fa_decode(q, k, v, o, lse, w.softmax_scale, n_ctas, ws)
    fa.fa_check_device_error(dev)
    n = per_config_steps(timed(3), steps)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(os.path.join("/tmp", f"fa_clocks_{os.getpid()}.csv")) as clocks:
        time.sleep(0.1)
        t = timed(n)
        time.sleep(0.1)
    fa.fa_check_device_error(dev)
    t = aggregate_over_ranks([t], world, dev)[0]
    peaks, peak_src = load_peaks()
    peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    achieved = algo_bytes / (t * 1e-3) / 1e9
    kname = f"decode_kt_kernel<{w.d}> (+ decode_merge_kernel<{w.d}>)"
    return {"config": {**config_of(w, world), "n_ctas": n_ctas}, "ms_per_step": t, "steps": n,
            "gbs": world * achieved,
            "roofline": {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": peak,
                         "unit": "GB/s", "frac": achieved / peak,
                         "peak_source": f"{peak_src} copy bandwidth",
                         "algorithmic_bytes": algo_bytes,
                         "traffic": recorded_traffic(kname, w)},
            "cpu_baseline": cpu, "gpu_launches": 2 * n, "clocks": clocks.summary(local)}


def run_decode(args, w, fa, inp, cpu, world, rank, local, dev, flush_buf):
    """Decoding: one fa_decode call per step (split kernel + merge kernel), the key/value cache
    resident in HBM. e2e: each step copies its new query rows from pinned host memory and reads
    O and lse back (the cache is state that stays on the device, not a per-step input)."""
    import numpy as np
    import torch
    import torch.distributed as dist
    from exact_attention_fa_gb300 import workloads as wl

    def dev_tensor(name):
        return torch.from_numpy(inp.raw(name).view(np.int16)).to(dev).view(torch.bfloat16)

    q, k, v = dev_tensor("q"), dev_tensor("k"), dev_tensor("v")
    scale = w.softmax_scale
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    n_ctas = fa.fa_decode_ctas(w.B, w.H, w.nq, w.N, w.d)
    ws = torch.empty(fa.fa_decode_workspace_bytes(w.B, w.H, w.nq, w.N, w.d), dtype=torch.uint8,
                     device=dev)
    algo_bytes = wl.decode_bytes(w)

    def step(qq=q, oo=o, ll=lse):
        fa.fa_decode(qq, k, v, oo, ll, scale, n_ctas, ws)

    for _ in range(args.warmup):
        flush_l2(flush_buf)
        step()
    fa.fa_check_device_error(dev)
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(os.path.join("/tmp", f"fa_clocks_{os.getpid()}.csv")) as clocks:
        time.sleep(0.1)
        t0 = time.perf_counter()
        for i in range(K):
            flush_l2(flush_buf)
            ev[i][0].record()
            step()
            ev[i][1].record()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        wall = time.perf_counter() - t0
        time.sleep(0.1)
    fa.fa_check_device_error(dev)
    t_step = statistics.fmean(ev[i][0].elapsed_time(ev[i][1]) for i in range(K))
    t_step = aggregate_over_ranks([t_step], world, dev)[0]

    e2e = None
    if not args.no_e2e:
        hq = q.cpu().pin_memory()
        ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        hl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        dq_, do_, dl_ = torch.empty_like(q), torch.empty_like(o), torch.empty_like(lse)
        E = min(K, 100)
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for i in range(E + 2):
            if i == 2:
                torch.cuda.synchronize()
                t_start.record()
            dq_.copy_(hq, non_blocking=True)
            step(dq_, do_, dl_)
            ho.copy_(do_, non_blocking=True)
            hl.copy_(dl_, non_blocking=True)
        t_end.record()
        torch.cuda.synchronize()
        fa.fa_check_device_error(dev)
        t_e2e = aggregate_over_ranks([t_start.elapsed_time(t_end) / E], world, dev)[0]
        e2e = {"value": world * algo_bytes / (t_e2e * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": hq.numel() * hq.element_size(),
               "d2h_bytes_per_step": ho.numel() * ho.element_size() + hl.numel() * hl.element_size(),
               "ms_per_step": t_e2e, "steps": E,
               "note": "key/value cache resident on the device; the step's new query rows go in, "
                       "O and lse come back"}
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    peaks, peak_src = load_peaks()
    peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    achieved = algo_bytes / (t_step * 1e-3) / 1e9
    kname = f"decode_kt_kernel<{w.d}> (+ decode_merge_kernel<{w.d}>)"
    line = {
        "metric": metric_name(w), "value": world * achieved, "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": t_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: i.i.d. N(0,1) inputs, seeded, rounded to bf16",
        "config": {**config_of(w, world), "n_ctas": n_ctas,
                   "l2": "flushed between steps outside the timed events (512 MiB write, then "
                          "256 MiB of it read back)"},
        "roofline": {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_src} copy bandwidth "
                                    f"{'MEASURED_PEAKS.json' if peak_src == 'measured' else 'fallback'}",
                     "frac_of_nominal": achieved / NOMINAL_HBM_GBS, "nominal": NOMINAL_HBM_GBS,
                     "algorithmic_bytes": algo_bytes,
                     "traffic": recorded_traffic(kname, w)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 2 * K,
        "clocks": clocks.summary(local),
        "wall_s_timed_region": wall,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
