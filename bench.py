#!/usr/bin/env python
"""Throughput of the exact-attention hot path on GB300 (one JSON line on stdout).

A step is one pass of the whole path over one batch: the tensor-core forward (O, lse) and, for
workloads with a backward, the recomputing backward (dQ, dK, dV) -- every launch goes through the
C ABI of libfa_gb300.so. The default workload is multi-head attention B=4, H=16, N=2048, d=64,
bf16, non-causal, forward + backward.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Metric: TFLOPS = algorithmic FLOPs / time, with 4*B*H*N^2*d for the forward (causal: half;
block-sparse: active tiles only) and 2.5 times that for the backward (its five contractions).
`value` is timed with CUDA events around the kernels only (inputs resident in HBM, L2 flushed
between steps by writing a 512 MiB buffer); `e2e` is the same step through the public API from
pinned host buffers, host<->device copies inside the timed region. Under torchrun every rank runs
its own replica of the workload (independent heads: no collective on the data path) and `value`
sums over ranks using the slowest rank's time.

Decoding workloads (decode_*: a few query rows per head against a long key/value cache) are
bound by HBM bandwidth, so their line reports GB/s of algorithmic bytes (K and V read once, q
read, O and lse written) against the measured copy bandwidth.

--impl reference times the fp64 CPU oracle (the parity reference) on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "mha_N2048_d64"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Datasheet figures for one GB300 (dense, no sparsity), reported beside the measured peaks.
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 7900.0
FP32_FMA_PER_CLK_PER_SM = 128  # fp32 FMA lanes per SM (four sub-partitions of 32)


def fp32_peak_tflops(peaks) -> float:
    """fp32 FMA peak from unit counts and clock: SMs x 128 FMA/clk x 2 FLOP x max SM clock."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    mhz = float(peaks.get("sm_max_mhz", 2070.0))
    return sms * FP32_FMA_PER_CLK_PER_SM * 2 * mhz * 1e6 / 1e12
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


def bench_workload(name: str):
    from exact_attention_fa_gb300 import workloads as wl
    w = wl.WORKLOADS[name]
    if name == DEFAULT_WORKLOAD:  # the default step is the whole path: forward + backward
        w = w.with_(backward=True)
    return w


def flops(w, mask=None):
    from exact_attention_fa_gb300 import workloads as wl
    f = wl.flop_count(w, mask, "fwd")
    return f, (2.5 * f if w.backward else 0.0)


def work_per_head(w, mask=None):
    """(amount of the metric's unit one (b, h) head represents, unit): TFLOP for attention
    steps, GB of algorithmic traffic for decoding."""
    from exact_attention_fa_gb300 import workloads as wl
    if w.decode:
        return wl.decode_bytes(w) / (w.B * w.H) / 1e9, "GB/s"
    f_fwd, f_bwd = flops(w, mask)
    return (f_fwd + f_bwd) / (w.B * w.H) / 1e12, "TFLOPS"


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


# ----------------------------------------------------------------------------------------- CPU

def oracle_tasks(w, inp, heads):
    mask = inp.raw("mask") if w.block_sparse else None
    tasks = []
    for idx in heads:
        b, h = divmod(idx % (w.B * w.H), w.H)
        do = inp.raw("do")[b, h] if w.backward else None
        tasks.append((inp.raw("q")[b, h], inp.raw("k")[b, h], inp.raw("v")[b, h], do,
                      w.softmax_scale, w.causal, mask))
    return tasks


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


def cpu_baseline_leg(w, inp, budget_s=20.0):
    """The oracle on a bounded sample of the workload's heads, on all host cores."""
    if w.dtype != "bf16":
        return None
    cores = host_cores()
    pool = make_pool(cores)
    try:
        per_head, unit = work_per_head(w, inp.raw("mask") if w.block_sparse else None)
        # one probe round of `cores` heads, then as many whole rounds as fit the budget
        n = min(cores, w.B * w.H)
        dt = time_oracle(pool, oracle_tasks(w, inp, range(n)))
        rounds = max(0, min(int(budget_s / max(dt, 1e-3)) - 1, (w.B * w.H) // n - 1))
        heads, total = n, dt
        if rounds:
            more = range(n, n + rounds * n)
            total += time_oracle(pool, oracle_tasks(w, inp, more))
            heads += len(more)
    finally:
        pool.terminate()
    return {"value": per_head * heads / total, "unit": unit, "cores": cores,
            "kind": "oracle",
            "sample": f"{heads} of {w.B * w.H} heads of {w.name}, fp64 numpy oracle "
                      f"({'forward+backward' if w.backward else 'forward'}), one head per worker",
            "seconds": round(total, 3)}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = bench_workload(args.workload)
    from exact_attention_fa_gb300 import workloads as wl
    inp = wl.make_inputs(w, with_do=w.backward)
    cores = host_cores()
    n = min(cores, w.B * w.H)
    per_head, unit = work_per_head(w, inp.raw("mask") if w.block_sparse else None)
    pool = make_pool(cores)
    times = []
    try:
        for i in range(args.warmup + args.steps):
            dt = time_oracle(pool, oracle_tasks(w, inp, range(i * n, (i + 1) * n)))
            if i >= args.warmup:
                times.append(dt)
    finally:
        pool.terminate()
    t = statistics.fmean(times)
    value = per_head * n / t
    sample = (f"{n} heads of {w.name} per step (one per worker), fp64 numpy oracle, "
              f"{'forward+backward' if w.backward else 'forward'}")
    print(json.dumps({
        "impl": "reference", "metric": metric_name(w), "value": value, "unit": unit,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args.gpus, note="oracle on host cores"),
        "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


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


def metric_name(w):
    if w.decode:
        return "attention decode GB/s (K, V read once; q, O, lse)"
    return "attention fwd/bwd TFLOPS (4·B·H·N²·d, causal halved)"


def config_of(w, n_gpus, note=None):
    c = {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "dtype": w.dtype,
         **({"Nq": w.nq, "Nk": w.N} if w.decode else {}),
         "causal": w.causal, "block_sparse": w.block_sparse,
         "step": "forward+backward" if w.backward else "forward",
         "global_batch": w.B * n_gpus, "seq_len": w.N, "parallelism": f"replicas{n_gpus}",
         "l2": "flushed between steps (512 MiB write)"}
    if note:
        c["note"] = note
    return c


# ----------------------------------------------------------------------------------------- GPU

class ClockSampler:
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
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
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
                for nm, val in zip(names[1:], parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = bench_workload(args.workload)
    from exact_attention_fa_gb300 import workloads as wl

    # host inputs first (and the oracle pool, if any, is spawned before CUDA is touched)
    inp = wl.make_inputs(w, with_do=w.backward)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_leg(w, inp)

    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import exact_attention_fa_gb300 as fa
    fa.load()

    def dev_tensor(name):
        a = inp.raw(name)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    q, k, v = dev_tensor("q"), dev_tensor("k"), dev_tensor("v")
    if w.decode:
        return run_decode(args, w, fa, q, k, v, cpu, world, rank, local, dev)
    do = dev_tensor("do") if w.backward else None
    mask = dev_tensor("mask") if w.block_sparse else None
    scale = w.softmax_scale
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    if w.backward:
        dq = torch.empty(q.shape, dtype=torch.float32, device=dev)
        dk, dv = torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.N, w.d), dtype=torch.uint8,
                         device=dev)
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def fwd():
        if w.dtype == "fp32":
            fa.fa_fwd_fp32(q, k, v, o, lse, scale, w.causal)
        elif w.block_sparse:
            fa.fa_fwd_blocksparse(q, k, v, o, lse, scale, mask)
        else:
            fa.fa_fwd(q, k, v, o, lse, scale, w.causal)

    def bwd():
        fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, scale, w.causal, ws)

    launches_per_step = (1 + (2 if w.backward else 0))
    f_fwd, f_bwd = flops(w, inp.raw("mask") if w.block_sparse else None)

    for _ in range(args.warmup):
        flush_buf.zero_()
        fwd()
        if w.backward:
            bwd()
    fa.fa_check_device_error(dev)

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(os.path.join("/tmp", f"fa_clocks_{os.getpid()}.csv")) as clocks:
        time.sleep(0.1)
        t0 = time.perf_counter()
        for i in range(K):
            flush_buf.zero_()
            ev[i][0].record()
            fwd()
            ev[i][1].record()
            if w.backward:
                bwd()
            ev[i][2].record()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        wall = time.perf_counter() - t0
        time.sleep(0.1)
    fa.fa_check_device_error(dev)
    step_ms = [ev[i][0].elapsed_time(ev[i][2]) for i in range(K)]
    fwd_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    bwd_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)] if w.backward else [0.0]
    t_step = statistics.fmean(step_ms)
    t_fwd = statistics.fmean(fwd_ms)
    t_bwd = statistics.fmean(bwd_ms)
    t_step, t_fwd, t_bwd = aggregate_over_ranks([t_step, t_fwd, t_bwd], world, dev)

    # ------------------------------------------------------------------ end to end, host buffers
    # Each step copies its inputs (Q, K, V and, with the backward, dO) from pinned host memory,
    # runs the step through the public API and reads every result back (O, lse and dQ, dK, dV).
    # Steps are pipelined the way a training loop prefetches: two sets of device buffers, the
    # host->device copy of step i+1 and the device->host copy of step i-1 run on their own
    # streams while step i computes. L2 is flushed before every step's compute, as above.
    e2e = None
    if not args.no_e2e:
        host_in = {n: t.cpu().pin_memory() for n, t in (("q", q), ("k", k), ("v", v))}
        if w.backward:
            host_in["do"] = do.cpu().pin_memory()
        out_names = ["o", "lse"] + (["dq", "dk", "dv"] if w.backward else [])
        proto = {"o": o, "lse": lse}
        if w.backward:
            proto.update(dq=dq, dk=dk, dv=dv)
        sets = []
        for _ in range(2):
            dev_in = {n: torch.empty_like(t, device=dev) for n, t in host_in.items()}
            dev_out = {n: torch.empty_like(proto[n]) for n in out_names}
            host_out = {n: torch.empty(proto[n].shape, dtype=proto[n].dtype, pin_memory=True)
                        for n in out_names}
            sets.append((dev_in, dev_out, host_out))
        ws2 = torch.empty_like(ws) if w.backward else None
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = sum(t.numel() * t.element_size() for t in sets[0][2].values())
        s_comp, s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def step_e2e(b):
            di, do_, _ = sets[b]
            if w.dtype == "fp32":
                fa.fa_fwd_fp32(di["q"], di["k"], di["v"], do_["o"], do_["lse"], scale, w.causal)
            elif w.block_sparse:
                fa.fa_fwd_blocksparse(di["q"], di["k"], di["v"], do_["o"], do_["lse"], scale, mask)
            else:
                fa.fa_fwd(di["q"], di["k"], di["v"], do_["o"], do_["lse"], scale, w.causal)
            if w.backward:
                fa.fa_bwd(di["q"], di["k"], di["v"], do_["o"], di["do"], do_["lse"], do_["dq"],
                          do_["dk"], do_["dv"], scale, w.causal, ws if b == 0 else ws2)

        E = min(K, 100)
        W2 = 2  # untimed pipelined steps first
        n_tot = W2 + E
        ev_in = [torch.cuda.Event() for _ in range(n_tot)]
        ev_comp = [torch.cuda.Event() for _ in range(n_tot)]
        ev_out = [torch.cuda.Event() for _ in range(n_tot)]
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        for i in range(n_tot):
            b = i % 2
            di, do_, ho = sets[b]
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
                flush_buf.zero_()
                step_e2e(b)
                ev_comp[i].record(s_comp)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(ev_comp[i])
                for n in out_names:
                    ho[n].copy_(do_[n], non_blocking=True)
                ev_out[i].record(s_d2h)
        s_d2h.wait_event(ev_out[n_tot - 1])
        t_end.record(s_d2h)
        torch.cuda.synchronize()
        fa.fa_check_device_error(dev)
        t_e2e = t_start.elapsed_time(t_end) / E
        t_e2e = aggregate_over_ranks([t_e2e], world, dev)[0]
        e2e = {"value": job_tflops(world, f_fwd + f_bwd, t_e2e), "unit": "TFLOPS",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e,
               "steps": E, "pipelined": "host->device, compute and device->host of consecutive "
                                        "steps overlap on three streams (two buffer sets)"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    # dominant kernel: the part of the step that takes longer
    if w.backward and t_bwd >= t_fwd:
        kname = f"bwd_tc_kernel<{w.d}> (+ bwd_prep_kernel<{w.d}> in the same call)"
        kflops, kms = f_bwd, t_bwd
    else:
        kname = forward_kernel_name(w)
        kflops, kms = f_fwd, t_fwd
    achieved = kflops / (kms * 1e-3) / 1e12
    peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    traffic = recorded_traffic(kname, w)
    if w.dtype == "fp32":  # the fp32 path runs on the FMA pipes, not the tensor cores
        alu_peak = fp32_peak_tflops(peaks)
        roofline = {"bound": "alu", "kernel": kname, "achieved": achieved, "peak": alu_peak,
                    "unit": "TFLOP/s", "frac": achieved / alu_peak,
                    "peak_source": "derived: SMs x 128 fp32 FMA/clk x 2 x max SM clock",
                    "traffic": traffic}
    else:
        roofline = {"bound": "tensor", "kernel": kname, "achieved": achieved, "peak": peak,
                    "unit": "TFLOP/s", "frac": achieved / peak,
                    "peak_source": f"{peak_src} bf16 dense (burst) "
                                   f"{'MEASURED_PEAKS.json' if peak_src == 'measured' else 'fallback'}",
                    "frac_of_sustained": achieved / sustained,
                    "frac_of_nominal": achieved / NOMINAL_BF16_TFLOPS,
                    "nominal": NOMINAL_BF16_TFLOPS,
                    "traffic": traffic}
    value = job_tflops(world, f_fwd + f_bwd, t_step)
    line = {
        "metric": metric_name(w), "value": value, "unit": "TFLOPS", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": t_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "fp32" if w.dtype == "fp32" else "bf16",
        "data": "synthetic: i.i.d. N(0,1) inputs, seeded" + (", rounded to bf16" if w.dtype == "bf16" else ""),
        "config": config_of(w, world),
        "parts": {
            "fwd": {"ms": t_fwd, "tflops": f_fwd / (t_fwd * 1e-3) / 1e12,
                    "frac_of_bf16_peak": f_fwd / (t_fwd * 1e-3) / 1e12 / peak},
            **({"bwd": {"ms": t_bwd, "tflops": f_bwd / (t_bwd * 1e-3) / 1e12,
                        "frac_of_bf16_peak": f_bwd / (t_bwd * 1e-3) / 1e12 / peak}}
               if w.backward else {}),
        },
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "clocks": clocks.summary(local),
        "wall_s_timed_region": wall,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_decode(args, w, fa, q, k, v, cpu, world, rank, local, dev):
    """Decoding: one fa_decode call per step (split kernel + merge kernel), the key/value cache
    resident in HBM. e2e: each step copies its new query rows from pinned host memory and reads
    O and lse back (the cache is state that stays on the device, not a per-step input)."""
    import torch
    import torch.distributed as dist
    from exact_attention_fa_gb300 import workloads as wl
    scale = w.softmax_scale
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    n_ctas = fa.fa_decode_ctas(w.B, w.H, w.nq, w.N, w.d)
    ws = torch.empty(fa.fa_decode_workspace_bytes(w.B, w.H, w.nq, w.N, w.d), dtype=torch.uint8,
                     device=dev)
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    algo_bytes = wl.decode_bytes(w)

    def step(qq=q, oo=o, ll=lse):
        fa.fa_decode(qq, k, v, oo, ll, scale, n_ctas, ws)

    for _ in range(args.warmup):
        flush_buf.zero_()
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
            flush_buf.zero_()
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
    kname = f"decode_stream_kernel<{w.d}> (+ decode_merge_kernel<{w.d}>)"
    line = {
        "metric": metric_name(w), "value": world * achieved, "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": t_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: i.i.d. N(0,1) inputs, seeded, rounded to bf16",
        "config": {**config_of(w, world), "n_ctas": n_ctas,
                   "l2": "inputs (K, V) larger than L2; also flushed between steps"},
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


def forward_kernel_name(w):
    """Name of the forward kernel the library runs for this workload (the two-query-tile kernel
    for every bf16 forward)."""
    if w.dtype == "fp32":
        return f"fwd_fp32_kernel<{w.d}>"
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
    entry = rec.get(f"{w.name}:{kname.split(' ')[0]}")
    if not entry or entry.get("source_digest") != build.source_digest():
        return None
    return entry.get("dram_bytes_per_launch")


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
