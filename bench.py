"""Benchmark of the attention hot path: one step = forward + backward through libfa.so.

Workload (the pages' benchmark family at 16k tokens per batch, head dim 128):
B=1, Hq=Hkv=16, N=16384, d=128, bf16 inputs iid N(0,1), scale=1/sqrt(d), non-causal.
FLOPs per step = 4*B*Hq*N^2*d (forward) * 3.5 (forward + backward at 2.5x forward),
halved for causal.  Prints ONE JSON line (see the keys below).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--causal] [--pass step|fwd|bwd]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

Multi-GPU: the path shards with no exchange step; under torchrun each rank runs an
independent replica of the workload ("weak" scaling), `value` sums all ranks' work over
the max-over-ranks time.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOP/s at 16k tokens/batch; % of GB300 BF16 tensor peak"
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--causal", action="store_true")
    ap.add_argument("--deterministic", action="store_true",
                    help="backward through fa_bwd_deterministic (fixed summation order)")
    ap.add_argument("--pass", dest="which", default="step", choices=["step", "fwd", "bwd"])
    ap.add_argument("--N", type=int, default=16384)
    ap.add_argument("--B", type=int, default=None)
    ap.add_argument("--H", type=int, default=16)
    ap.add_argument("--Hkv", type=int, default=None, help="key/value heads (default: --H, i.e. MHA)")
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--varlen", action="store_true",
                    help="packed variable-length batch of --N tokens (default 16384): sequence lengths drawn "
                         "uniformly from [--min-len, --max-len] with a fixed seed")
    ap.add_argument("--decode", action="store_true",
                    help="decode forward: --B sequences (default 8) of --N cached keys (default 16384), "
                         "--Nq new queries, Hq=--H (default 32 here), Hkv=--Hkv (default 8 here)")
    ap.add_argument("--paged", action="store_true",
                    help="with --decode: the caches as 128-row pages in a shuffled order behind a block table")
    ap.add_argument("--fp8", action="store_true",
                    help="forward only with E4M3 q, k, v (per-tensor descales), bf16 output")
    ap.add_argument("--block-scales", action="store_true",
                    help="with --fp8: one descale per 128-row block of each head (fa_fwd_fp8_blockscaled)")
    ap.add_argument("--Nq", type=int, default=1)
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--min-len", type=int, default=512)
    ap.add_argument("--max-len", type=int, default=4096)
    return ap.parse_args()


def workload(a):
    B = a.B if a.B is not None else max(1, 16384 // a.N)
    Hkv = a.Hkv if a.Hkv is not None else a.H
    return dict(B=B, Hq=a.H, Hkv=Hkv, N=a.N, d=a.d, causal=bool(a.causal), dtype="bf16",
                deterministic=bool(getattr(a, "deterministic", False)))


def flops(w, which):
    f = 4.0 * w["B"] * w["Hq"] * w["N"] ** 2 * w["d"]
    if w["causal"]:
        f /= 2
    return {"fwd": f, "bwd": 2.5 * f, "step": 3.5 * f}[which]


def workload_name(w, which):
    passes = {"step": "fwd+bwd", "fwd": "fwd", "bwd": "bwd"}[which]
    return (f"exact attention {passes}, B={w['B']} Hq={w['Hq']} Hkv={w['Hkv']} N={w['N']} d={w['d']} "
            f"{w['dtype']} {'causal' if w['causal'] else 'non-causal'} ({w['B'] * w['N'] // 1024}k tokens/batch)"
            + (", deterministic backward" if w.get("deterministic") else ""))


def kernel_source_digest(kernel):
    """sha256 of the sources that define `kernel` (its .cu file and the shared headers)."""
    import hashlib

    csrc = os.path.join(ROOT, "exact_attention_38_gb300", "csrc")
    files = {"fa_fwd_kernel": ["fa_fwd.cu", "fa_math.cuh", "exp2_poly.h"],
             "fa_bwd_main": ["fa_bwd.cu", "fa_bwd_common.cuh"]}[kernel]
    h = hashlib.sha256()
    for f in files + ["sm100_ptx.cuh", "fa_internal.h"]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu record, or None when the kernel's
    sources changed since the counters were taken (or the workload differs)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel)
    if not rec or rec.get("source_sha256") != kernel_source_digest(kernel) or rec.get("workload") != workload:
        return None
    return rec.get("bytes_per_launch")


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return j.get("bf16_tflops"), j.get("hbm_gbs"), "measured"
    return 1900.0, 6800.0, "fallback"


# ------------------------------------------------------- multi-rank aggregation

def reduce_step_time(ms_local, world, device=None):
    """Max over ranks of the per-step time (every rank runs its own replica)."""
    if world <= 1:
        return float(ms_local)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(ms_local)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank_step, world, ms_step):
    """Whole-job TFLOP/s: the work of all ranks over the slowest rank's step time."""
    return world * flops_per_rank_step / (ms_step * 1e-3) / 1e12


# ------------------------------------------------------------- host cost per call

def host_us_per_call(fn, reps=50):
    """Median host time of one call (argument checks, tensor-map encoding, launches),
    measured with the GPU idle: the device is synchronised before every call, and the
    call returns once its kernels are enqueued.  Includes the Python-to-C (ctypes)
    marshalling of the call."""
    import torch

    ts = []
    for _ in range(reps):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        fn()
        ts.append(time.perf_counter() - t0)
    torch.cuda.synchronize()
    return statistics.median(ts) * 1e6


def ctypes_floor_us(fa, reps=200):
    """Median time of a call into the library that does nothing (fa_status_string): the
    marshalling part of the per-call figures."""
    ts = []
    for _ in range(reps):
        t0 = time.perf_counter()
        fa.lib.fa_status_string(0)
        ts.append(time.perf_counter() - t0)
    return statistics.median(ts) * 1e6


# ----------------------------------------------------------- clocks during timing

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ CPU baseline

def host_cpu():
    """Host CPU description for the baseline record (architecture and model, if known)."""
    import platform

    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                key = ln.split(":")[0].strip().lower()
                if key in ("model name", "cpu part", "hardware"):
                    model = ln.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return f"{platform.machine()} {model}".strip()


def cpu_oracle_sample(w, steps=1, target_s=12.0):
    """The fp64 oracle, as it stands, on a bounded slice of the same workload: the first
    n_s positions of `heads` heads, sized from a short calibration run so one step takes
    about `target_s` seconds of host time (at most the workload's N and Hq)."""
    import numpy as np

    import oracle
    from exact_attention_38_gb300.inputs import make_inputs, to_f64

    cores = len(os.sched_getaffinity(0))
    scale = 1.0 / math.sqrt(w["d"])
    # calibration: one head, 1024 positions (the oracle's cost grows as heads * N^2)
    n_c = min(w["N"], 1024)
    xc = {k: to_f64(v) for k, v in make_inputs(1, n_c, 1, 1, w["d"], dtype=w["dtype"], seed=4).items()}
    t0 = time.perf_counter()
    oracle.attn_bwd_ref(xc["q"], xc["k"], xc["v"], xc["do"], w["causal"], scale)
    per_head_c = max(time.perf_counter() - t0, 1e-4)
    n_s = w["N"]
    while n_s > n_c and per_head_c * (n_s / n_c) ** 2 > target_s:
        n_s //= 2
    heads = int(max(1, min(w["Hq"], round(target_s / (per_head_c * (n_s / n_c) ** 2)))))
    x = make_inputs(1, n_s, heads, heads, w["d"], dtype=w["dtype"], seed=3)
    xo = {k: to_f64(v) for k, v in x.items()}
    fl = 3.5 * 4.0 * heads * n_s ** 2 * w["d"] * (0.5 if w["causal"] else 1.0)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        r = oracle.attn_bwd_ref(xo["q"], xo["k"], xo["v"], xo["do"], w["causal"], scale)
        times.append(time.perf_counter() - t0)
        assert np.isfinite(r["dq"]).all()
    sample = (f"oracle attn_bwd_ref (fwd+all grads, fp64 numpy) on B=1, {heads} heads, N={n_s}, d={w['d']} "
              f"({'causal' if w['causal'] else 'non-causal'}), sized for ~{target_s:.0f} s per step; FLOPs by the "
              f"same formula")
    return fl, times, cores, sample


def run_reference(a):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = workload(a)
    # every step a bounded sample, sized so the whole run stays within about two minutes
    per_step = max(0.5, min(12.0, 120.0 / max(1, a.warmup + a.steps)))
    fl, times, cores, sample = cpu_oracle_sample(w, steps=a.warmup + a.steps, target_s=per_step)
    t = times[a.warmup:] if len(times) > a.warmup else times
    sec = sum(t) / len(t)
    val = fl / sec / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": a.gpus,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(w, "step") + " [oracle runs a bounded slice, see cpu_baseline]",
                       "parallelism": "host cores"},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample,
                             "cpu": host_cpu(), "seconds_per_step": sec},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------- native

def run_native(a):
    import torch
    import torch.distributed as dist

    from exact_attention_38_gb300 import fa
    from exact_attention_38_gb300.inputs import make_inputs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = workload(a)
    B, Hq, Hkv, N, d, causal = w["B"], w["Hq"], w["Hkv"], w["N"], w["d"], w["causal"]
    scale = 1.0 / math.sqrt(d)
    x = make_inputs(B, N, Hq, Hkv, d, dtype=w["dtype"], seed=3 + rank)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = fa.fa_bwd_workspace_size(B, Hq, Hkv, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    DT = fa.FA_BF16

    def fwd():
        st = fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, Hq, Hkv, N, d,
                       causal, scale, DT, sp)
        if st != fa.FA_OK:
            raise fa.FaError(st, "fa_fwd")

    bwd_fn = fa.fa_bwd_deterministic if a.deterministic else fa.fa_bwd

    def bwd():
        st = bwd_fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                    dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, N, d, causal, scale, DT,
                    ws.data_ptr(), ws_bytes, sp)
        if st != fa.FA_OK:
            raise fa.FaError(st, bwd_fn.__name__)

    parts = {"step": [("fwd", fwd), ("bwd", bwd)], "fwd": [("fwd", fwd)], "bwd": [("bwd", bwd)]}[a.which]
    if a.which == "bwd":
        fwd()
    # backward: preprocess, key-block kernel, dQ convert (deterministic: dQ kernel), plus the
    # wave-tail split's dK / dV convert when the one-CTA-per-key-block grid is split (the
    # library's rule: non-causal, N > 512, last wave at most half of the SMs)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    units = B * Hkv * ((N + 127) // 128)
    split = (not causal and N > 512 and 0 < units % sms <= sms // 2
             and (units % sms) * 2 * 128 * d * 4 <= B * N * Hq * d * 2)
    launches_per_step = sum({"fwd": 1, "bwd": 4 if split else 3}[n] for n, _ in parts)

    for _ in range(a.warmup):
        for _, fn in parts:
            fn()
    torch.cuda.synchronize()
    fa.check_device_error()

    K = a.steps
    ev = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
          for n, _ in parts}
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        time.sleep(0.3)
        t_wall = time.perf_counter()
        for i in range(K):
            flush.zero_()  # evict the previous step's data from L2 (outside the events)
            for n, fn in parts:
                ev[n][i][0].record(stream)
                fn()
                ev[n][i][1].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    fa.check_device_error()
    host_us = {"fa_fwd": host_us_per_call(fwd), bwd_fn.__name__: host_us_per_call(bwd),
               "ctypes_floor": ctypes_floor_us(fa),
               "how": "median over 50 calls, GPU idle (synchronised before each call), ctypes marshalling included"}
    per = {n: [e0.elapsed_time(e1) for e0, e1 in ev[n]] for n in ev}
    ms_step = reduce_step_time(sum(statistics.mean(per[n]) for n in per), world, dev)
    if world > 1:
        dist.barrier()
    fl_step = flops(w, a.which)
    value = job_throughput(fl_step, world, ms_step)

    # ---- e2e: host buffers through the C ABI, copies inside the timed region.  Two sets
    # of device buffers and two copy streams pipeline the steps the way a serving loop
    # would: step i+1's inputs are copied in and step i-1's results copied out while
    # step i computes; every step's copies are still inside the timed region.
    e2e = None
    if not a.no_e2e:
        hq, hk, hv, hdo = (t.cpu().pin_memory() for t in (x["q"], x["k"], x["v"], x["do"]))
        host_out = [[torch.empty_like(t, device="cpu").pin_memory() for t in (q, lse, q, k, v)] for _ in range(2)]
        sets = [dict(q=q, k=k, v=v, do=do, o=o, lse=lse, dq=dq, dk=dk, dv=dv, ws=ws)]
        sets.append({n: torch.empty_like(t) for n, t in sets[0].items()})
        sets[1]["o"].copy_(o)
        sets[1]["lse"].copy_(lse)  # the bwd-only pass reads the forward's outputs

        def c_step(bf):
            if a.which in ("step", "fwd"):
                st_ = fa.fa_fwd(bf["q"].data_ptr(), bf["k"].data_ptr(), bf["v"].data_ptr(), bf["o"].data_ptr(),
                                bf["lse"].data_ptr(), B, Hq, Hkv, N, d, causal, scale, DT, sp)
                if st_ != fa.FA_OK:
                    raise fa.FaError(st_, "fa_fwd")
            if a.which in ("step", "bwd"):
                st_ = bwd_fn(bf["q"].data_ptr(), bf["k"].data_ptr(), bf["v"].data_ptr(), bf["o"].data_ptr(),
                             bf["lse"].data_ptr(), bf["do"].data_ptr(), bf["dq"].data_ptr(), bf["dk"].data_ptr(),
                             bf["dv"].data_ptr(), B, Hq, Hkv, N, d, causal, scale, DT, bf["ws"].data_ptr(), ws_bytes,
                             sp)
                if st_ != fa.FA_OK:
                    raise fa.FaError(st_, bwd_fn.__name__)

        in_names = ["q", "k", "v", "do"] if a.which != "fwd" else ["q", "k", "v"]
        out_names = ["o", "lse", "dq", "dk", "dv"] if a.which != "fwd" else ["o", "lse"]
        h_in = dict(q=hq, k=hk, v=hv, do=hdo)
        h2d = sum(h_in[n].numel() * h_in[n].element_size() for n in in_names)
        d2h = sum(sets[0][n].numel() * sets[0][n].element_size() for n in out_names)
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for rep in range(2):
            torch.cuda.synchronize()
            e0.record(stream)
            s_in.wait_event(e0)
            done_out = [None, None]
            for i in range(K):
                bf, ho = sets[i % 2], host_out[i % 2]
                if done_out[i % 2] is not None:
                    s_in.wait_event(done_out[i % 2])  # the set's previous results are out
                with torch.cuda.stream(s_in):
                    for n in in_names:
                        bf[n].copy_(h_in[n], non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
                stream.wait_event(ev_in)
                c_step(bf)
                ev_c = torch.cuda.Event()
                ev_c.record(stream)
                s_out.wait_event(ev_c)
                with torch.cuda.stream(s_out):
                    for hdst, n in zip(ho, out_names):
                        hdst.copy_(bf[n], non_blocking=True)
                done_out[i % 2] = torch.cuda.Event()
                done_out[i % 2].record(s_out)
            ev_last = torch.cuda.Event()
            ev_last.record(s_out)
            stream.wait_event(ev_last)
            e1.record(stream)
            torch.cuda.synchronize()
        ms_e2e = reduce_step_time(e0.elapsed_time(e1) / K, world, dev)
        e2e = {"value": job_throughput(fl_step, world, ms_e2e), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
               "pipelining": "two device buffer sets; inputs of step i+1 copied in and results of step i-1 "
                             "copied out on two copy streams while step i computes"}
        fa.check_device_error()

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peak_tf, peak_hbm, peak_kind = measured_peaks()
    # dominant kernel: the pass with the largest share of the step
    dom = max(per, key=lambda n: statistics.mean(per[n]))
    dom_ms = statistics.mean(per[dom])
    achieved = flops(w, dom) / (dom_ms * 1e-3) / 1e12
    if dom == "fwd":
        # fa_fwd runs its persistent kernel for N <= 512 (N <= 1024 with the mask)
        short = w["N"] <= (1024 if w.get("causal") else 512)
        kern, timed = ("fa_fwd_persistent" if short else "fa_fwd_kernel"), "one fa_fwd call (one launch)"
    elif w.get("deterministic"):
        # the key-block kernel is the persistent one for N <= 512
        kb = "fa_bwd_persistent" if w["N"] <= 512 else "fa_bwd_main"
        kern = kb + "+fa_bwd_dq_kernel"
        timed = (f"one fa_bwd_deterministic call: preprocess + {kb} without its dQ path + fa_bwd_dq_kernel "
                 "(FLOPs by the 2.5x backward count; the two kernels execute 3.5x the forward's)")
    else:
        kern = "fa_bwd_persistent" if w["N"] <= 512 else "fa_bwd_main"
        timed = (f"one fa_bwd call: preprocess + {kern} + dQ convert (the key-block kernel is ~98% of it at "
                 "16k-token sequences, ~72% at N=512)")
    roofline = {"bound": "tensor", "kernel": kern, "timed": timed,
                "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s", "frac": achieved / peak_tf,
                "traffic": (recorded_traffic(kern, workload_name(w, "step"))
                            if kern in ("fa_fwd_kernel", "fa_bwd_main") else None),
                "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)",
                "peak_kind": f"{peak_kind} bf16 dense, burst (of measured)"}
    passes = {n: {"ms": statistics.mean(per[n]), "ms_min": min(per[n]),
                  "tflops": flops(w, n) / (statistics.mean(per[n]) * 1e-3) / 1e12} for n in per}
    for n in passes:
        passes[n]["frac_of_peak"] = passes[n]["tflops"] / peak_tf

    cpu = None
    if not a.no_cpu_baseline:
        fl_s, times, cores, sample = cpu_oracle_sample(w, steps=1)
        cpu = {"value": fl_s / times[0] / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": sample, "seconds": times[0], "cpu": host_cpu()}

    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": a.warmup,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload_name(w, a.which), "B": B, "Hq": Hq, "Hkv": Hkv, "N": N, "d": d,
                       "causal": causal, "global_batch": B * world, "seq_len": N,
                       "parallelism": f"replicas x{world} (no exchange step)",
                       "l2": "flushed between steps (2x L2 buffer written outside the timed events); "
                             "inputs (q,k,v,dO,o = 320 MiB) also exceed L2"},
            "passes": passes, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches_per_step * K, "wall_s_timed_region": t_wall, "host_us_per_call": host_us,
            "clocks": clk.summary()}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------- variable-length batches

def varlen_lengths(total, lo, hi, seed=7):
    """Sequence lengths drawn uniformly from [lo, hi] (Python's seeded generator) until
    `total` tokens are reached; the last one is cut to fit."""
    import random

    rng = random.Random(seed)
    lens = []
    while sum(lens) < total:
        lens.append(rng.randint(lo, hi))
    lens[-1] -= sum(lens) - total
    return [n for n in lens if n > 0]


def visible_pairs(nq, nk, causal):
    """(query, key) pairs the mask leaves visible; the mask is aligned at the
    bottom-right corner (query i sees key j iff j <= i + nk - nq)."""
    if not causal:
        return nq * nk
    return sum(max(0, min(nk, i + nk - nq + 1)) for i in range(nq))


def run_varlen(a):
    import torch

    from exact_attention_38_gb300 import fa
    from exact_attention_38_gb300.inputs import make_varlen_inputs

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    total = a.N
    lens = varlen_lengths(total, a.min_len, a.max_len)
    Hq = a.H
    Hkv = a.Hkv if a.Hkv is not None else a.H
    d, causal = a.d, bool(a.causal)
    x = make_varlen_inputs(lens, lens, Hq, Hkv, d, dtype="bf16", seed=3)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    cu = x["cu_q"].to(dev)
    mx = max(lens)
    scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q)
    lse = torch.empty((Hq, total), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = fa.fa_bwd_varlen_workspace_size(len(lens), Hq, mx, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    sp = torch.cuda.current_stream(dev).cuda_stream
    B = len(lens)

    def fwd():
        st = fa.fa_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), cu.data_ptr(),
                              cu.data_ptr(), None, None, B, Hq, Hkv, total, total, mx, mx, d, causal, scale,
                              fa.FA_BF16, sp)
        if st != fa.FA_OK:
            raise fa.FaError(st, "fa_fwd_varlen")

    def bwd():
        st = fa.fa_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                              dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), cu.data_ptr(), cu.data_ptr(), None, None,
                              B, Hq, Hkv, total, total, mx, mx, d, causal, scale, fa.FA_BF16, ws.data_ptr(),
                              ws_bytes, sp)
        if st != fa.FA_OK:
            raise fa.FaError(st, "fa_bwd_varlen")

    for _ in range(a.warmup):
        fwd()
        bwd()
    torch.cuda.synchronize()
    fa.check_device_error()
    ev = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
          for n in ("fwd", "bwd")}
    stream = torch.cuda.current_stream(dev)
    with ClockSampler(0) as clk:
        time.sleep(0.3)
        for i in range(a.steps):
            flush.zero_()
            for n, fn in (("fwd", fwd), ("bwd", bwd)):
                ev[n][i][0].record(stream)
                fn()
                ev[n][i][1].record(stream)
        torch.cuda.synchronize()
    fa.check_device_error()
    ms = {n: statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev[n]) for n in ev}
    f_fwd = sum(4.0 * Hq * d * visible_pairs(n, n, causal) for n in lens)
    fl = {"fwd": f_fwd, "bwd": 2.5 * f_fwd}
    peak_tf, _, peak_kind = measured_peaks()
    passes = {n: {"ms": ms[n], "tflops": fl[n] / (ms[n] * 1e-3) / 1e12} for n in ms}
    for n in passes:
        passes[n]["frac_of_peak"] = passes[n]["tflops"] / peak_tf
    ms_step = ms["fwd"] + ms["bwd"]
    value = (fl["fwd"] + fl["bwd"]) / (ms_step * 1e-3) / 1e12
    dom = max(ms, key=ms.get)
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"exact attention fwd+bwd, packed variable-length batch of {total} tokens: "
                                   f"{B} sequences, lengths uniform in [{a.min_len}, {a.max_len}] (seed 7), "
                                   f"Hq={Hq} Hkv={Hkv} d={d} bf16 {'causal' if causal else 'non-causal'}",
                       "lengths": lens, "l2": "flushed between steps (outside the timed events)"},
            "passes": passes,
            "roofline": {"bound": "tensor", "kernel": "fa_fwd_kernel" if dom == "fwd" else "fa_bwd_main",
                         "achieved": passes[dom]["tflops"], "peak": peak_tf, "unit": "TFLOP/s",
                         "frac": passes[dom]["tflops"] / peak_tf, "traffic": None,
                         "peak_kind": f"{peak_kind} bf16 dense, burst (of measured)"},
            "cpu_baseline": None, "e2e": None, "gpu_launches": 4 * a.steps, "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def run_decode(a):
    import torch

    from exact_attention_38_gb300 import fa
    from exact_attention_38_gb300.inputs import make_decode_inputs

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    B = a.B if a.B is not None else 8
    Hq = a.H if a.H != 16 else 32  # the GQA shape of the long-context configuration by default
    Hkv = a.Hkv if a.Hkv is not None else 8
    N, Nq, d, causal = a.N, a.Nq, a.d, bool(a.causal)
    x = make_decode_inputs(B, Nq, N, Hq, Hkv, d, dtype="bf16", seed=3)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    cl = torch.full((B,), N, dtype=torch.int32, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
    S = fa.fa_decode_num_splits(B, Hq, Hkv, Nq, N, d, a.splits)
    ws_bytes = fa.fa_decode_workspace_size(B, Hq, Hkv, Nq, N, d, a.splits)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    # evicted by READING a buffer twice the size of L2: a written flush would leave up to
    # a whole L2 of dirty lines whose write-back lands inside the next timed decode, which
    # itself writes almost nothing
    flush = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    sp = torch.cuda.current_stream(dev).cuda_stream
    scale = 1.0 / math.sqrt(d)

    def step():
        st = fa.fa_fwd_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), cl.data_ptr(), o.data_ptr(), lse.data_ptr(),
                              B, Hq, Hkv, Nq, N, d, causal, scale, a.splits, fa.FA_BF16, ws.data_ptr(), ws_bytes, sp)
        if st != fa.FA_OK:
            raise fa.FaError(st, "fa_fwd_decode")

    if a.paged:
        # the same caches cut into 128-row pages stored in a shuffled order
        P = (N + 127) // 128
        g = torch.Generator().manual_seed(5)
        perm = torch.randperm(B * P, generator=g).to(dev)
        table = perm.view(B, P).to(torch.int32).contiguous()

        def to_pages(c):
            padded = torch.zeros((B, P * 128, Hkv, d), dtype=c.dtype, device=dev)
            padded[:, :N] = c
            pages = torch.empty((B * P, 128, Hkv, d), dtype=c.dtype, device=dev)
            pages[perm] = padded.view(B * P, 128, Hkv, d)
            return pages

        kp, vp = to_pages(k), to_pages(v)
        del k, v
        ws_bytes = fa.fa_decode_workspace_size(B, Hq, Hkv, Nq, P * 128, d, a.splits)
        ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)

        def step():  # noqa: F811
            st = fa.fa_fwd_decode_paged(q.data_ptr(), kp.data_ptr(), vp.data_ptr(), table.data_ptr(), cl.data_ptr(),
                                        o.data_ptr(), lse.data_ptr(), B, Hq, Hkv, Nq, B * P, P, d, causal, scale,
                                        a.splits, fa.FA_BF16, ws.data_ptr(), ws_bytes, sp)
            if st != fa.FA_OK:
                raise fa.FaError(st, "fa_fwd_decode_paged")

    for _ in range(a.warmup):
        step()
    torch.cuda.synchronize()
    fa.check_device_error()
    stream = torch.cuda.current_stream(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
    with ClockSampler(0) as clk:
        time.sleep(0.3)
        for i in range(a.steps):
            flush.sum()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    fa.check_device_error()
    host_us = {"fa_fwd_decode_paged" if a.paged else "fa_fwd_decode": host_us_per_call(step),
               "ctypes_floor": ctypes_floor_us(fa),
               "how": "median over 50 calls, GPU idle (synchronised before each call), ctypes marshalling included"}
    ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)
    # algorithmic bytes: every cached key and value row once, q read, o and lse written
    kv_bytes = 2 * B * N * Hkv * d * 2
    io_bytes = 2 * B * Nq * Hq * d * 2 + 4 * B * Hq * Nq
    gbs = (kv_bytes + io_bytes) / (ms * 1e-3) / 1e9
    _, peak_hbm, peak_kind = measured_peaks()
    pairs = sum(visible_pairs(Nq, N, causal) for _ in range(B))
    tflops = 4.0 * Hq * d * pairs / (ms * 1e-3) / 1e12
    line = {"metric": "decode: KV-cache bytes read per second", "value": gbs, "unit": "GB/s", "n_gpus": 1,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"exact attention decode forward: B={B} sequences x {N} cached keys, Nq={Nq} new "
                                   f"queries, Hq={Hq} Hkv={Hkv} d={d} bf16 {'causal' if causal else 'non-causal'}, "
                                   f"{S} key splits{', paged cache (128-row pages, shuffled)' if a.paged else ''}",
                       "l2": "flushed between steps by reading a 2x L2 buffer (outside the timed events; no "
                             "dirty lines left); the cache exceeds L2"},
            "tflops": tflops,
            "roofline": {"bound": "hbm", "kernel": "fa_decode_kernel (+ fa_decode_combine)", "achieved": gbs,
                         "peak": peak_hbm, "unit": "GB/s", "frac": gbs / peak_hbm, "traffic": None,
                         "bytes_per_step": kv_bytes + io_bytes, "peak_kind": f"{peak_kind} HBM copy (of measured)"},
            "cpu_baseline": None, "e2e": None, "gpu_launches": (2 if S > 1 else 1) * a.steps,
            "host_us_per_call": host_us, "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def run_fp8(a):
    import torch

    from exact_attention_38_gb300 import fa
    from exact_attention_38_gb300.inputs import make_fp8_block_inputs, make_fp8_inputs

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    w = workload(a)
    B, Hq, Hkv, N, d, causal = w["B"], w["Hq"], w["Hkv"], w["N"], w["d"], w["causal"]
    blk = bool(getattr(a, "block_scales", False))
    x = make_fp8_block_inputs(B, N, Hq, Hkv, d, seed=3) if blk else make_fp8_inputs(B, N, Hq, Hkv, d, seed=3)
    bs = {n: x[n + "_descale"].to(dev) for n in ("q", "k", "v")} if blk else None
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    ws_bytes = fa.fa_fwd_fp8_workspace_size(B, Hkv, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    sp = torch.cuda.current_stream(dev).cuda_stream
    scale = 1.0 / math.sqrt(d)

    def fwd():
        if blk:
            st = fa.fa_fwd_fp8_blockscaled(q.data_ptr(), k.data_ptr(), v.data_ptr(), bs["q"].data_ptr(),
                                           bs["k"].data_ptr(), bs["v"].data_ptr(), o.data_ptr(), lse.data_ptr(), B, Hq,
                                           Hkv, N, d, causal, scale, ws.data_ptr(), ws_bytes, sp)
        else:
            st = fa.fa_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, Hq, Hkv, N,
                               d, causal, scale, x["q_descale"], x["k_descale"], x["v_descale"], ws.data_ptr(),
                               ws_bytes, sp)
        if st != fa.FA_OK:
            raise fa.FaError(st, "fa_fwd_fp8")

    for _ in range(a.warmup):
        fwd()
    torch.cuda.synchronize()
    fa.check_device_error()
    stream = torch.cuda.current_stream(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
    with ClockSampler(0) as clk:
        time.sleep(0.3)
        for i in range(a.steps):
            flush.zero_()
            ev[i][0].record(stream)
            fwd()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    fa.check_device_error()
    ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)
    tf = flops(w, "fwd") / (ms * 1e-3) / 1e12
    peak_bf16, _, peak_kind = measured_peaks()
    peak = 2.0 * peak_bf16  # E4M3 dense rate = 2 x bf16 (nominal 4.5 / 2.25 PFLOP/s)
    line = {"metric": METRIC, "value": tf, "unit": "TFLOP/s", "n_gpus": 1, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
            "data": "synthetic",
            "config": {"workload": workload_name(w, "fwd").replace(
                "bf16", "e4m3 in (descales per 128-row block and head), bf16 out" if blk else "e4m3 in, bf16 out"),
                       "l2": "flushed between steps (outside the timed events)"},
            "roofline": {"bound": "tensor", "kernel": "fa_fwd_fp8_kernel (+ V transpose)", "achieved": tf,
                         "peak": peak, "unit": "TFLOP/s", "frac": tf / peak, "traffic": None,
                         "peak_kind": f"{peak_kind} bf16 burst x 2 (E4M3 / bf16 nominal ratio)"},
            "cpu_baseline": None, "e2e": None, "gpu_launches": 2 * a.steps, "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def main():
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    elif a.fp8:
        run_fp8(a)
    elif a.decode:
        run_decode(a)
    elif a.varlen:
        run_varlen(a)
    else:
        run_native(a)


if __name__ == "__main__":
    main()
