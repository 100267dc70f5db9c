#!/usr/bin/env python3
"""Benchmark of the exact-attention hot path on GB300.

One step = one pass of the whole path over one batch of synthetic inputs:
  * prefill: FlashAttention-2 forward, B=1 H=32 Sq=Sk=4096 D=128 bf16, causal
    (the LLaMA-7B prefill shape of the pages' benchmark table), and
  * decode: split-KV decoding, B=16 H=8 Sk=8192 D=128 bf16, 32 partitions,
    phase 1 + log-sum-exp merge in one launch (the last partition of each head
    merges it); the two-launch form (phase 1, then a merge launch) is timed
    beside it.
The headline `value` is prefill attention TFLOPS (causal FLOPs counted at half
of 4*B*H*S^2*D); the decode throughput in GB/s (K and V read once, plus q and
O) sits in the `decode` object. Inputs are resident in HBM, and L2 is flushed
(a 256 MiB write) before every step, outside the timed kernels. Each kernel is
timed with CUDA events on the stream it is launched on. After the timed loop,
a sustained leg runs the prefill kernel back to back for about a second with
the SM clock sampled (`sustained_prefill`), next to the short loop's figure.

`--impl reference` times the fp64 CPU oracle instead (a bounded sample of the
same workload per step) with the same metric and unit.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
For N > 1 launch under torchrun: every rank runs its own replica of the
workload (no data-path communication; weak scaling) and rank 0 reports the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attn fwd TFLOPS & % bf16 tensor peak; split-KV decode HBM GB/s & % peak"
PREFILL = "llama_prefill"
DECODE = "decode"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# The sources each captured kernel is compiled from: a committed DRAM-traffic
# figure is reported only while these still hash to the captured ones.
_CSRC = "exact_attention_54_gb300/csrc/"
KERNEL_SOURCES = {
    "fa_fwd_kernel": [_CSRC + "fa_fwd_kernel.cuh", _CSRC + "sm103_ptx.cuh", _CSRC + "fa_launch.h"],
    "fa_decode_split_kernel_fused": [_CSRC + "fa_decode.cu", _CSRC + "fa_launch.h"],
    "fa_splitkv_merge_kernel": [_CSRC + "fa_decode.cu", _CSRC + "fa_launch.h"],
    "fa_fwd_d256_kernel": [_CSRC + "fa_fwd_d256.cuh", _CSRC + "sm103_ptx.cuh", _CSRC + "fa_launch.h"],
    "fa_fwd_d256_kernel_d512": [_CSRC + "fa_fwd_d256.cuh", _CSRC + "sm103_ptx.cuh", _CSRC + "fa_launch.h"],
    "fa_fwd_d256_kernel_d1024": [_CSRC + "fa_fwd_d256.cuh", _CSRC + "sm103_ptx.cuh", _CSRC + "fa_launch.h"],
    "fa_bwd_kernel": [_CSRC + "fa_bwd.cuh", _CSRC + "sm103_ptx.cuh", _CSRC + "fa_launch.h"],
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=50, help="steps of the end-to-end (host buffer) loop")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU time of the oracle baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end loop (profiling runs)")
    ap.add_argument("--sustained-seconds", type=float, default=1.0,
                    help="kernel seconds of the back-to-back prefill leg (0 skips it)")
    ap.add_argument("--parts", default="prefill,decode",
                    help="comma list of the path parts to run (profiling runs may isolate one: prefill, decode, "
                         "backward, d256, splitd, varlen, varlen_backward, shapes, decode_two, paged)")
    return ap.parse_args(argv)


# ------------------------------------------------------------- environment --

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS if k in p}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic():
    """Per-launch DRAM bytes from the committed ncu captures, for each kernel
    whose sources still hash to the captured ones (others are left out)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return {}
    with open(path) as f:
        t = json.load(f)
    out = {}
    for name, rec in t.get("kernels", {}).items():
        if name in KERNEL_SOURCES and rec.get("hash") == kernel_source_hash(name):
            out[name] = rec.get("bytes")
    return out


def aggregate_max(values, world):
    """Element-wise max over ranks (timings: the slowest rank decides)."""
    if world == 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64)
    if dist.get_backend() == "nccl":
        t = t.cuda()
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.cpu().tolist()


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed loop runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu), "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def _snapshot(self):
        try:
            out = subprocess.run(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                  "-i", str(self.gpu)], capture_output=True, text=True, timeout=20).stdout
            return [ln for ln in out.splitlines() if ln.strip()]
        except (OSError, subprocess.SubprocessError):
            return []

    def stop(self, t_begin: float, t_end: float):
        """Summarise the samples stamped inside [t_begin, t_end] (time.time())."""
        import datetime
        lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=10)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            with open(self.path) as f:
                lines = [ln for ln in f.read().splitlines() if ln.strip()]
        if self.path:
            os.unlink(self.path)
        source = "during"
        if not lines:
            lines, source = self._snapshot(), "after"
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        inside = []
        for ln in lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                ts = None
            inside.append((ts is not None and t_begin <= ts <= t_end, f))
        if source == "during" and any(ok for ok, _ in inside):
            rows = [f for ok, f in inside if ok]
        else:  # no sample fell inside the loop: keep what there is, and say so
            rows = [f for _, f in inside]
            if source == "during":
                source = "around"
        for f in rows:
            try:
                sm.append(float(f[2]))
                mx.append(float(f[3]))
            except ValueError:
                continue
            try:
                pw.append(float(f[4]))
            except ValueError:
                pass
            for name, val in zip(names, f[6:10]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "when": source}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "when": source, "power_w_max": max(pw) if pw else None}


# ------------------------------------------------------------------ oracle --

_INPUT_CACHE = {}


def _cached_inputs(w):
    from exact_attention_54_gb300 import inputs
    if w.name not in _INPUT_CACHE:
        _INPUT_CACHE[w.name] = inputs.make_workload(w)
    return _INPUT_CACHE[w.name]


def oracle_rate(w, target_s: float, threads: int | None = None):
    """Time the fp64 oracle, as it stands, on a bounded sample of workload w:
    one head per host thread (all host cores unless `threads` is given), a
    strided subset of query rows in each. Returns (TFLOPS of useful attention
    work, threads, description, seconds)."""
    import oracle
    from exact_attention_54_gb300 import inputs
    from exact_attention_54_gb300.metrics import attention_flops

    threads = threads or oracle.default_threads()
    heads = min(threads, w.B * w.H)
    q, k, v = _cached_inputs(w)
    q = q.reshape(-1, w.Sq, w.D)[:heads]
    k = k.reshape(-1, w.Sk, w.D)[:heads]
    v = v.reshape(-1, w.Sk, w.D)[:heads]

    def useful(rows):
        keys = [min(r + 1, w.Sk) if w.causal else w.Sk for r in rows]
        return sum(4.0 * n * w.D for n in keys) * heads

    probe = list(range(0, w.Sq, max(1, w.Sq // 8)))[:8]
    t0 = time.perf_counter()
    oracle.attention(q, k, v, w.causal, w.scale, rows=probe, nthreads=threads)
    per_row = (time.perf_counter() - t0) / len(probe)
    n = int(max(1, min(w.Sq, target_s / max(per_row, 1e-9))))
    stride = max(1, w.Sq // n)
    rows = list(range(0, w.Sq, stride))[:n]
    t0 = time.perf_counter()
    oracle.attention(q, k, v, w.causal, w.scale, rows=rows, nthreads=threads)
    dt = time.perf_counter() - t0
    assert attention_flops(1, 1, w.Sq, w.Sk, w.D, w.causal) > 0
    desc = (f"{heads} of {w.B * w.H} heads x {len(rows)} of {w.Sq} query rows (stride {stride}) of {w.name}; "
            f"fp64, S and P materialised per row; untuned C oracle")
    return useful(rows) / dt / 1e12, threads, desc, dt


def oracle_decode_rate(w, target_s: float):
    """fp64 oracle on a bounded sample of the decode workload (heads x all keys),
    as GB/s of the K/V bytes the sample covers."""
    import oracle
    from exact_attention_54_gb300 import inputs

    threads = oracle.default_threads()
    q, k, v = _cached_inputs(w)
    q = q.reshape(-1, 1, w.D)
    k = k.reshape(-1, w.Sk, w.D)
    v = v.reshape(-1, w.Sk, w.D)
    t0 = time.perf_counter()
    oracle.attention(q[:threads], k[:threads], v[:threads], False, w.scale, nthreads=threads)
    per_head = (time.perf_counter() - t0) / min(threads, q.shape[0])
    heads = int(max(1, min(q.shape[0], target_s / max(per_head, 1e-9))))
    t0 = time.perf_counter()
    oracle.attention(q[:heads], k[:heads], v[:heads], False, w.scale, nthreads=threads)
    dt = time.perf_counter() - t0
    nbytes = heads * (2 * w.Sk * w.D + 2 * w.D) * 2
    return nbytes / dt / 1e9, threads, f"{heads} of {q.shape[0]} heads of {w.name} (all keys), fp64 oracle", dt


def run_reference(args, rank, world):
    """The reference arm: the fp64 oracle on the host cores, same metric/unit."""
    if rank != 0:
        return None
    from exact_attention_54_gb300 import inputs
    w = inputs.WORKLOADS[PREFILL]
    budget = min(10.0, 120.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_rate(w, budget)
    rates, secs = [], []
    desc, threads = "", 1
    for _ in range(args.steps):
        r, threads, desc, dt = oracle_rate(w, budget)
        rates.append(r)
        secs.append(dt)
    value = statistics.median(rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(),
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
                         "sample": f"per step: {desc}"},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


def config_block():
    return {"workload": "llama7b_prefill_b1h32s4096d128_bf16_causal + decode_b16h8sk8192d128_bf16_split32",
            "prefill": {"B": 1, "H": 32, "Sq": 4096, "Sk": 4096, "D": 128, "dtype": "bf16", "causal": True,
                        "scale": "1/sqrt(128)"},
            "decode": {"B": 16, "H": 8, "Sq": 1, "Sk": 8192, "D": 128, "dtype": "bf16", "num_splits": 32},
            "l2": "flushed before every step (256 MiB write, outside the timed kernels)",
            "inputs": "seeded i.i.d. N(0,1), resident in HBM"}


# --------------------------------------------------------------------- GPU --

def run_gpu(args, rank, world, local):
    import torch

    import exact_attention_54_gb300 as fa
    from exact_attention_54_gb300 import inputs
    from exact_attention_54_gb300.metrics import attention_flops, decode_bytes

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    fa.load_library()

    wp = inputs.WORKLOADS[PREFILL]
    wd = inputs.WORKLOADS[DECODE]
    parts = set(args.parts.split(","))
    run_pf, run_dc = "prefill" in parts, "decode" in parts
    full = run_pf and run_dc  # the report; a profiling run of some parts allocates only what they use
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    if run_pf or "backward" in parts:
        q, k, v = (t.to(dev) for t in inputs.make_workload(wp))
        o = torch.empty_like(q)
        lse = torch.empty(wp.B, wp.H, wp.Sq, dtype=torch.float32, device=dev)
    if run_dc or "decode_two" in parts:
        dq, dk, dv = (t.to(dev) for t in inputs.make_workload(wd))
        S = wd.num_splits
        ws = (torch.empty(wd.B, wd.H, S, wd.D, dtype=torch.float32, device=dev),
              torch.empty(wd.B, wd.H, S, dtype=torch.float32, device=dev),
              torch.empty(wd.B, wd.H, S, dtype=torch.float32, device=dev))
        counters = torch.zeros(wd.B * wd.H, dtype=torch.int32, device=dev)
        do = torch.empty(wd.B, wd.H, 1, wd.D, dtype=wd.dtype, device=dev)
        dlse = torch.empty(wd.B, wd.H, dtype=torch.float32, device=dev)

    pf_flops = attention_flops(wp.B, wp.H, wp.Sq, wp.Sk, wp.D, wp.causal)
    dc_bytes = decode_bytes(wd.B, wd.H, wd.Sk, wd.D)

    if parts & {"backward", "d256", "splitd", "varlen", "varlen_backward", "shapes", "decode_two", "paged"} and \
            not (run_pf or run_dc):
        # profiling run of the backward pass or of the large-head forwards alone
        rec = {"part": args.parts, "steps": args.steps}
        if "backward" in parts:
            rec["backward"] = run_bwd(args, fa, torch, stream, dev, flush, world, (q, k, v), o, lse, wp)
        if "d256" in parts:
            rec["d256_prefill"] = run_wide_head(args, fa, torch, dev, stream, flush, world, "d256")
        if "splitd" in parts:
            rec["split_d"] = {key: run_wide_head(args, fa, torch, dev, stream, flush, world, key)
                              for key in ("large_head", "massive_head")}
        if "varlen" in parts:
            rec["varlen_prefill"] = run_varlen(args, fa, torch, dev, stream, flush, world)
            rec["small_prefill"] = run_wide_head(args, fa, torch, dev, stream, flush, world, "small")
        if "varlen_backward" in parts:
            rec["varlen_backward"] = run_varlen_bwd(args, fa, torch, dev, stream, flush, world)
        if "paged" in parts:
            rec["paged_decode"] = run_paged(args, fa, torch, stream, dev, flush, world)
        if "shapes" in parts:
            rec["shapes"] = run_shapes(args, fa, torch, dev, stream, flush, world)
        if "decode_two" in parts:
            rec["decode_two_launch"] = run_two_launch(args, fa, torch, stream, flush, world, (dq, dk, dv), ws, do,
                                                      dlse, wd)
        if rank == 0:
            print(json.dumps(rec), flush=True)
        return None

    def step(evs=None):
        flush.fill_(float(1.0))
        if evs:
            evs[0].record(stream)
        if run_pf:
            fa.fa_fwd(q, k, v, o, lse, wp.causal, wp.scale, stream)
        if evs:
            evs[1].record(stream)
        if run_dc:
            fa.fa_decode_splitkv_fused(dq, dk, dv, do, dlse, *ws, counters, S, wd.scale, stream)
        if evs:
            evs[2].record(stream)

    # one untimed pass checks the device error word before anything is timed
    step()
    torch.cuda.synchronize()
    fa.fa_check_device_error()

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)  # nvidia-smi start-up; samples before t_begin are discarded
    # the W warm-up steps run right before the timed ones, so that the timed
    # region does not start on a GPU that has just idled for the sampler
    for _ in range(args.warmup):
        step()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    t_begin = time.time()
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(events[i])
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    t_end = time.time()
    if world > 1:
        dist.barrier()
    clock = clocks.stop(t_begin, t_end)
    fa.fa_check_device_error()

    pf = [e[0].elapsed_time(e[1]) for e in events]  # ms
    dc = [e[1].elapsed_time(e[2]) for e in events]
    pf_sum, dc_sum, wall = aggregate_max([sum(pf), sum(dc), wall], world)
    K = args.steps

    if not full:  # a profiling run of one part: a short record, not the report
        rec = {"part": args.parts, "steps": args.steps, "clocks": clock}
        if run_pf:
            rec.update(prefill_tflops=pf_flops / (statistics.mean(pf) * 1e-3) / 1e12,
                       prefill_ms=statistics.mean(pf), prefill_ms_median=statistics.median(pf))
        if run_dc:
            rec.update(decode_gbs=dc_bytes / (statistics.mean(dc) * 1e-3) / 1e9, decode_ms=statistics.mean(dc))
        if rank == 0:
            print(json.dumps(rec), flush=True)
        return None
    prefill_tflops = world * pf_flops * K / (pf_sum * 1e-3) / 1e12
    decode_gbs = world * dc_bytes * K / (dc_sum * 1e-3) / 1e9
    two = run_two_launch(args, fa, torch, stream, flush, world, (dq, dk, dv), ws, do, dlse, wd)
    d256 = run_wide_head(args, fa, torch, dev, stream, flush, world, "d256")
    split_d = {key: run_wide_head(args, fa, torch, dev, stream, flush, world, key)
               for key in ("large_head", "massive_head")}
    varlen = run_varlen(args, fa, torch, dev, stream, flush, world)
    small = run_wide_head(args, fa, torch, dev, stream, flush, world, "small")
    bwd = run_bwd(args, fa, torch, stream, dev, flush, world, (q, k, v), o, lse, wp)
    varlen_bwd = run_varlen_bwd(args, fa, torch, dev, stream, flush, world)
    paged = run_paged(args, fa, torch, stream, dev, flush, world)
    sustained = (None if args.sustained_seconds <= 0 else
                 run_sustained(args, fa, torch, stream, flush, world, local, (q, k, v), o, lse, wp,
                               statistics.mean(pf)))
    # end-to-end through host buffers (pinned), copies inside the timed region
    e2e = ({"prefill": None, "decode": None} if args.no_e2e else
           run_e2e(args, fa, torch, stream, dev, wp, wd, (q, k, v), (dq, dk, dv), world))

    peaks, peak_src = load_peaks()
    traffic = committed_traffic()
    pf_avg_ms = statistics.mean(pf)
    dc_avg_ms = statistics.mean(dc)
    achieved_tf = pf_flops / (pf_avg_ms * 1e-3) / 1e12
    achieved_gbs = dc_bytes / (dc_avg_ms * 1e-3) / 1e9
    tb = traffic.get("fa_fwd_kernel")
    line = {
        "metric": METRIC, "value": prefill_tflops, "unit": "TFLOPS", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": (pf_sum + dc_sum) / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_block(),
        "roofline": {"bound": "tensor", "kernel": "fa_fwd_kernel<128,bf16,causal>", "achieved": achieved_tf,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved_tf / peaks["bf16_tflops"],
                     "traffic": tb, "peak_source": f"{peak_src} bf16 dense (burst)",
                     "frac_of_sustained": achieved_tf / peaks["bf16_tflops_sustained"],
                     "per_launch_flops": pf_flops, "avg_launch_ms": pf_avg_ms},
        "decode": {
            "metric": "split-KV decode HBM GB/s", "value": decode_gbs, "unit": "GB/s",
            "ms_per_step": dc_sum / K, "path": "fa_decode_splitkv_fused (phase 1 + merge, one launch)",
            "roofline": {"bound": "hbm", "kernel": "fa_decode_split_kernel<128,bf16,dense,fused>",
                         "achieved": achieved_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved_gbs / peaks["hbm_gbs"], "frac_of_8000_nominal": achieved_gbs / 8000.0,
                         "traffic": traffic.get("fa_decode_split_kernel_fused"), "peak_source": f"{peak_src} copy",
                         "per_step_bytes": dc_bytes, "avg_launch_ms": dc_avg_ms},
            "two_launch": two,
            "e2e": e2e["decode"],
        },
        "e2e": e2e["prefill"],
        "decode_gbs": decode_gbs,
        "decode_frac": achieved_gbs / peaks["hbm_gbs"],
        "sustained_prefill": sustained,
        "paged_decode": paged,
        "d256_prefill": d256,
        "split_d": split_d,
        "varlen_prefill": varlen,
        "small_prefill": small,
        "backward": bwd,
        "varlen_backward": varlen_bwd,
        "gpu_launches": 2 * K,
        "clocks": clock,
        "wall_ms_per_step": 1e3 * wall / K,
    }
    return line


def run_sustained(args, fa, torch, stream, flush, world, local, qkv, o, lse, wp, launch_ms):
    """The prefill kernel back to back for at least --sustained-seconds of
    kernel time (L2 flushed before every launch, as in the timed loop), each
    launch timed with CUDA events, the SM clock and power sampled throughout:
    the steady-state figure beside the short timed loop. kcycles_per_launch =
    time x median SM clock, to compare runs at different clocks."""
    from exact_attention_54_gb300.metrics import attention_flops
    q, k, v = qkv
    n = max(10, int(math.ceil(args.sustained_seconds / (launch_ms * 1e-3))))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    clocks = ClockSampler(local)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_begin = time.time()
    for a, b in evs:
        flush.fill_(float(1.0))
        a.record(stream)
        fa.fa_fwd(q, k, v, o, lse, wp.causal, wp.scale, stream)
        b.record(stream)
    torch.cuda.synchronize()
    t_end = time.time()
    clock = clocks.stop(t_begin, t_end)
    fa.fa_check_device_error()
    ms = aggregate_max([statistics.mean(a.elapsed_time(b) for a, b in evs)], world)[0]
    flops = attention_flops(wp.B, wp.H, wp.Sq, wp.Sk, wp.D, wp.causal)
    peaks, src = load_peaks()
    tf = world * flops / (ms * 1e-3) / 1e12
    mhz = clock.get("sm_mhz")
    return {"value": tf, "unit": "TFLOPS", "launches": n, "kernel_seconds": n * ms * 1e-3, "ms_per_launch": ms,
            "frac_of_sustained_peak": tf / peaks["bf16_tflops_sustained"],
            "frac_of_burst_peak": tf / peaks["bf16_tflops"], "peak_source": src, "clocks": clock,
            "kcycles_per_launch": (ms * 1e-3 * mhz * 1e6 / 1e3) if mhz else None}


def run_two_launch(args, fa, torch, stream, flush, world, dec, ws, o, lse, wd):
    """The two-launch decode (fa_decode_splitkv, then fa_splitkv_merge) on the
    decode workload, timed on its own loop with the same L2 flush."""
    from exact_attention_54_gb300.metrics import decode_bytes
    dq, dk, dv = dec
    S = wd.num_splits
    n = max(1, min(args.steps, 500))

    def step(evs=None):
        flush.fill_(float(1.0))
        if evs:
            evs[0].record(stream)
        fa.fa_decode_splitkv(dq, dk, dv, *ws, S, wd.scale, stream)
        if evs:
            evs[1].record(stream)
        fa.fa_splitkv_merge(*ws, o, lse, stream)
        if evs:
            evs[2].record(stream)

    for _ in range(3):
        step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    for i in range(n):
        step(evs[i])
    torch.cuda.synchronize()
    sp, mg = aggregate_max([sum(e[0].elapsed_time(e[1]) for e in evs) / n,
                            sum(e[1].elapsed_time(e[2]) for e in evs) / n], world)
    nbytes = decode_bytes(wd.B, wd.H, wd.Sk, wd.D)
    peaks, _ = load_peaks()
    gbs = world * nbytes / ((sp + mg) * 1e-3) / 1e9
    return {"value": gbs, "unit": "GB/s", "split_ms": sp, "merge_ms": mg, "steps": n,
            "frac_of_hbm": gbs / peaks["hbm_gbs"], "split_only_gbs": world * nbytes / (sp * 1e-3) / 1e9,
            "traffic_merge": committed_traffic().get("fa_splitkv_merge_kernel")}


def run_bwd(args, fa, torch, stream, dev, flush, world, qkv, o, lse, wp):
    """Backward pass on the prefill workload (causal LLaMA-7B shape, bf16),
    dO seeded like the inputs; the three launches of fa_bwd timed together
    on their own loop with the same L2 flush. FLOPs: 2.5x the forward's (five
    products of the same size instead of two), causal at half."""
    from exact_attention_54_gb300 import inputs
    from exact_attention_54_gb300.metrics import attention_flops
    q, k, v = qkv
    fa.fa_fwd(q, k, v, o, lse, wp.causal, wp.scale, stream)
    do = inputs.make_dense(wp.B, wp.H, wp.Sq, wp.Sq, wp.D, wp.dtype, seed=wp.seed + 100)[0].to(dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(wp.B, wp.H, wp.Sq, wp.D) // 4, dtype=torch.float32, device=dev)
    n = max(1, min(args.steps, 300))

    def step(evs=None):
        flush.fill_(float(1.0))
        if evs:
            evs[0].record(stream)
        fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, wp.causal, wp.scale, stream)
        if evs:
            evs[1].record(stream)

    for _ in range(3):
        step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for i in range(n):
        step(evs[i])
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    ms = aggregate_max([sum(e[0].elapsed_time(e[1]) for e in evs) / n], world)[0]
    flops = 2.5 * attention_flops(wp.B, wp.H, wp.Sq, wp.Sk, wp.D, wp.causal)
    peaks, _ = load_peaks()
    tf = world * flops / (ms * 1e-3) / 1e12
    return {"workload": wp.name, "value": tf, "unit": "TFLOPS", "ms_per_call": ms, "steps": n,
            "launches_per_call": 3, "frac_of_bf16_peak": tf / peaks["bf16_tflops"], "per_call_flops": flops,
            "traffic_main_kernel": committed_traffic().get("fa_bwd_kernel")}


def run_wide_head(args, fa, torch, dev, stream, flush, world, key):
    """A dense forward workload timed on its own loop with the same L2 flush:
    the pages' large-head rows, fp16, non-causal ("GPT-4 style" (1, 16, 2048,
    2048, 256) on the 256-column kernel, "Large Head" (1, 8, 1024, 1024, 512)
    and "Massive Head" (1, 4, 512, 512, 1024) on its Split-D form) and the
    small (8, 16, 256, 256, 64) case. TFLOPS count the attention FLOPs
    (4 B H Sq Sk D); Split-D also executes Q K^T once per 256-column output
    slice, reported as executed_tflops."""
    from exact_attention_54_gb300 import inputs
    from exact_attention_54_gb300.metrics import attention_flops
    w = inputs.WORKLOADS[key]
    q, k, v = (t.to(dev) for t in inputs.make_workload(w))
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.Sq, dtype=torch.float32, device=dev)
    n = max(1, min(args.steps, 500))

    def step(evs=None):
        flush.fill_(float(1.0))
        if evs:
            evs[0].record(stream)
        fa.fa_fwd(q, k, v, o, lse, w.causal, w.scale, stream)
        if evs:
            evs[1].record(stream)

    for _ in range(3):
        step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for i in range(n):
        step(evs[i])
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    ms = aggregate_max([sum(e[0].elapsed_time(e[1]) for e in evs) / n], world)[0]
    flops = attention_flops(w.B, w.H, w.Sq, w.Sk, w.D, w.causal)
    slices = max(1, w.D // 256)
    executed = flops * (slices + 1) / 2 if slices > 1 else flops
    peaks, src = load_peaks()
    tf = world * flops / (ms * 1e-3) / 1e12
    kernel = (f"fa_fwd_d256_kernel<{w.D},fp16,non-causal,dense>" if w.D >= 256 else
              f"fa_fwd_kernel<{w.D},fp16,non-causal,dense>")
    rec = {"workload": w.name, "value": tf, "unit": "TFLOPS", "ms_per_launch": ms, "steps": n,
           "kernel": kernel, "frac_of_bf16_peak": tf / peaks["bf16_tflops"], "per_launch_flops": flops}
    if key == "small":
        rec.update(short_launch_context(args, fa, torch, dev, stream, flush, world, w, n))
    if w.D < 256:
        return rec
    if slices > 1:
        rec.update(output_slices=slices, executed_tflops=world * executed / (ms * 1e-3) / 1e12)
    rec["traffic"] = committed_traffic().get("fa_fwd_d256_kernel" + (f"_d{w.D}" if slices > 1 else ""))
    return rec


def short_launch_context(args, fa, torch, dev, stream, flush, world, w, n):
    """Context for a launch this short (a few microseconds of work per CTA):
    - launch_floor_us: an empty kernel with the forward's launch shape (128
      CTAs of 384 threads, 166,656 bytes of dynamic shared memory), timed
      the same way (L2 flushed, events around the one launch): the fixed
      cost of any launch of that shape;
    - back_to_back: the forward launched 400 times in a row over 40 input
      sets used in turn (336 MB, more than L2, so no flush between them),
      one event pair around all of them: the rate of a stream of such
      calls, where one launch's set-up overlaps the previous one's drain."""
    import ctypes
    from exact_attention_54_gb300 import build as fabuild
    from exact_attention_54_gb300.metrics import attention_flops
    st = ctypes.CDLL(fabuild.SELFTEST_LIB)
    st.fa_selftest_empty_launch.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    sp = stream.cuda_stream

    def empty():
        if st.fa_selftest_empty_launch(128, 384, 166656, sp) != 0:
            raise RuntimeError("fa_selftest_empty_launch failed")

    for _ in range(3):
        flush.fill_(float(1.0))
        empty()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for i in range(n):
        flush.fill_(float(1.0))
        evs[i][0].record(stream)
        empty()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    floor_ms = aggregate_max([sum(e[0].elapsed_time(e[1]) for e in evs) / n], world)[0]

    from exact_attention_54_gb300 import inputs
    sets = []
    for i in range(40):
        q, k, v = (t.to(dev) for t in inputs.make_workload(w))
        sets.append((q, k, v, torch.empty_like(q), torch.empty(w.B, w.H, w.Sq, dtype=torch.float32, device=dev)))
    launches = 400
    for i in range(40):
        fa.fa_fwd(*sets[i][:4], sets[i][4], w.causal, w.scale, stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush.fill_(float(1.0))
    e0.record(stream)
    for i in range(launches):
        q, k, v, o, lse = sets[i % 40]
        fa.fa_fwd(q, k, v, o, lse, w.causal, w.scale, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    b2b_ms = aggregate_max([e0.elapsed_time(e1) / launches], world)[0]
    flops = attention_flops(w.B, w.H, w.Sq, w.Sk, w.D, w.causal)
    del sets
    return {"launch_floor_us": floor_ms * 1e3,
            "back_to_back": {"us_per_launch": b2b_ms * 1e3, "tflops": world * flops / (b2b_ms * 1e-3) / 1e12,
                             "launches": launches, "input_sets": 40}}


def run_shapes(args, fa, torch, dev, stream, flush, world):
    """Context rows outside the default run: the LLaMA-7B shape without the
    causal mask and the pages' BERT-large shape (8, 32, 2048, 2048, 128),
    bf16, seeded N(0,1) inputs; each timed like the prefill (L2 flushed,
    CUDA events per launch)."""
    from exact_attention_54_gb300 import inputs
    from exact_attention_54_gb300.metrics import attention_flops
    shapes = {"llama7b_noncausal": (1, 32, 4096, 128, False), "bert_large_noncausal": (8, 32, 2048, 128, False),
              "bert_large_causal": (8, 32, 2048, 128, True)}
    peaks, _ = load_peaks()
    out = {}
    n = max(1, min(args.steps, 300))
    for name, (B, H, S, D, causal) in shapes.items():
        q, k, v = (t.to(dev) for t in inputs.make_dense(B, H, S, S, D, torch.bfloat16, seed=2024))
        o = torch.empty_like(q)
        lse = torch.empty(B, H, S, dtype=torch.float32, device=dev)

        def step(evs=None):
            flush.fill_(float(1.0))
            if evs:
                evs[0].record(stream)
            fa.fa_fwd(q, k, v, o, lse, causal, D ** -0.5, stream)
            if evs:
                evs[1].record(stream)

        for _ in range(3):
            step()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        for i in range(n):
            step(evs[i])
        torch.cuda.synchronize()
        fa.fa_check_device_error()
        ms = aggregate_max([sum(e[0].elapsed_time(e[1]) for e in evs) / n], world)[0]
        tf = world * attention_flops(B, H, S, S, D, causal) / (ms * 1e-3) / 1e12
        out[name] = {"shape": [B, H, S, S, D], "causal": causal, "ms_per_launch": ms, "value": tf, "unit": "TFLOPS",
                     "frac_of_bf16_peak": tf / peaks["bf16_tflops"]}
        del q, k, v, o, lse
    return out


def run_varlen(args, fa, torch, dev, stream, flush, world):
    """The pages' packed-sequence row: 16 sequences with lengths drawn
    uniformly from [64, 2048], [T, 16, 128] bf16, causal, int32 cu_seqlens.
    TFLOPS count sum_i 2 H L_i^2 D (the causal half of 4 H L_i^2 D); timed
    on its own loop with the same L2 flush."""
    from exact_attention_54_gb300 import inputs
    from exact_attention_54_gb300.metrics import varlen_flops
    w = inputs.WORKLOADS["varlen"]
    lengths, cu, q, k, v = inputs.make_workload(w)
    q, k, v, cu = (t.to(dev) for t in (q, k, v, cu.to(torch.int32)))
    o = torch.empty_like(q)
    lse = torch.empty(w.H, q.shape[0], dtype=torch.float32, device=dev)
    max_len = int(lengths.max())
    n = max(1, min(args.steps, 500))

    def step(evs=None):
        flush.fill_(float(1.0))
        if evs:
            evs[0].record(stream)
        fa.fa_fwd_varlen(q, k, v, o, lse, cu, cu, max_len, w.causal, w.scale, stream)
        if evs:
            evs[1].record(stream)

    for _ in range(3):
        step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for i in range(n):
        step(evs[i])
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    ms = aggregate_max([sum(e[0].elapsed_time(e[1]) for e in evs) / n], world)[0]
    flops = varlen_flops(lengths.tolist(), lengths.tolist(), w.H, w.D, w.causal)
    peaks, _ = load_peaks()
    tf = world * flops / (ms * 1e-3) / 1e12
    return {"workload": w.name, "value": tf, "unit": "TFLOPS", "ms_per_launch": ms, "steps": n,
            "kernel": "fa_fwd_kernel<128,bf16,causal,varlen>", "frac_of_bf16_peak": tf / peaks["bf16_tflops"],
            "per_launch_flops": flops, "total_tokens": int(q.shape[0]), "max_seqlen": max_len}


def run_varlen_bwd(args, fa, torch, dev, stream, flush, world):
    """Backward pass over the packed-sequence workload (16 sequences of
    64-2048 tokens, H16 D128 bf16, causal), dO seeded like the inputs; the
    three launches of fa_bwd_varlen timed together with the same L2 flush.
    FLOPs: 2.5x the forward's count (five products of its size)."""
    from exact_attention_54_gb300 import inputs
    from exact_attention_54_gb300.metrics import varlen_flops
    w = inputs.WORKLOADS["varlen"]
    lengths, cu, q, k, v = inputs.make_workload(w)
    do = inputs.make_varlen(w.num_seqs, 0, 0, w.H, w.D, w.dtype, seed=w.seed + 100, lengths=lengths.tolist())[2]
    q, k, v, do, cu = (t.to(dev) for t in (q, k, v, do, cu))
    mx = int(lengths.max())
    o, lse = fa.flash_attention_varlen(q, k, v, cu, cu, mx, causal=w.causal, scale=w.scale, stream=stream)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_varlen_workspace_bytes(q.shape[0], w.H, w.D) // 4, dtype=torch.float32, device=dev)
    n = max(1, min(args.steps, 300))

    def step(evs=None):
        flush.fill_(float(1.0))
        if evs:
            evs[0].record(stream)
        fa.fa_bwd_varlen(q, k, v, o, do, lse, dq, dk, dv, ws, cu, cu, mx, mx, w.causal, w.scale, stream)
        if evs:
            evs[1].record(stream)

    for _ in range(3):
        step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for i in range(n):
        step(evs[i])
    torch.cuda.synchronize()
    fa.fa_check_device_error()
    ms = aggregate_max([sum(e[0].elapsed_time(e[1]) for e in evs) / n], world)[0]
    flops = 2.5 * varlen_flops(lengths.tolist(), lengths.tolist(), w.H, w.D, w.causal)
    peaks, _ = load_peaks()
    tf = world * flops / (ms * 1e-3) / 1e12
    return {"workload": w.name, "value": tf, "unit": "TFLOPS", "ms_per_call": ms, "steps": n,
            "launches_per_call": 3, "frac_of_bf16_peak": tf / peaks["bf16_tflops"], "per_call_flops": flops}


def run_paged(args, fa, torch, stream, dev, flush, world):
    """Split-KV decode over a paged cache (16-key pages, permuted block table),
    same shapes and bytes as the decode workload; timed on its own loop with
    the same L2 flush and CUDA events, one-launch (fused) and two-launch."""
    from exact_attention_54_gb300 import inputs
    from exact_attention_54_gb300.metrics import decode_bytes
    w = inputs.WORKLOADS["paged_decode"]
    q, kc, vc, bt, sl = (t.to(dev) for t in inputs.make_workload(w))
    S = w.num_splits
    ws = (torch.empty(w.B, w.H, S, w.D, dtype=torch.float32, device=dev),
          torch.empty(w.B, w.H, S, dtype=torch.float32, device=dev),
          torch.empty(w.B, w.H, S, dtype=torch.float32, device=dev))
    o = torch.empty(w.B, w.H, 1, w.D, dtype=w.dtype, device=dev)
    lse = torch.empty(w.B, w.H, dtype=torch.float32, device=dev)
    counters = torch.zeros(w.B * w.H, dtype=torch.int32, device=dev)
    n = max(1, min(args.steps, 500))

    def step(fused, evs=None):
        flush.fill_(float(1.0))
        if evs:
            evs[0].record(stream)
        if fused:
            fa.fa_decode_paged_splitkv_fused(q, kc, vc, bt, sl, o, lse, *ws, counters, S, w.scale, stream)
        else:
            fa.fa_decode_paged_splitkv(q, kc, vc, bt, sl, *ws, S, w.scale, stream)
            fa.fa_splitkv_merge(*ws, o, lse, stream)
        if evs:
            evs[1].record(stream)

    res = {}
    for fused in (True, False):
        for _ in range(3):
            step(fused)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        for i in range(n):
            step(fused, evs[i])
        torch.cuda.synchronize()
        fa.fa_check_device_error()
        res[fused] = aggregate_max([sum(e[0].elapsed_time(e[1]) for e in evs) / n], world)[0]
    nbytes = decode_bytes(w.B, w.H, w.Sk, w.D)
    peaks, src = load_peaks()
    gbs = world * nbytes / (res[True] * 1e-3) / 1e9
    gbs2 = world * nbytes / (res[False] * 1e-3) / 1e9
    return {"workload": w.name, "value": gbs, "unit": "GB/s", "ms_per_step": res[True], "steps": n,
            "path": "fa_decode_paged_splitkv_fused", "frac_of_hbm": gbs / peaks["hbm_gbs"],
            "block_size": w.extra["block_size"],
            "two_launch": {"value": gbs2, "unit": "GB/s", "ms_per_step": res[False],
                           "frac_of_hbm": gbs2 / peaks["hbm_gbs"]}}


def run_e2e(args, fa, torch, stream, dev, wp, wd, pre, dec, world):
    """Same metrics through the public API from pinned host buffers: every step
    copies its inputs host->device, runs the kernels and reads the outputs back.
    Steps are pipelined the way a serving loop would run them: two sets of
    device and host buffers, the host->device copies on one stream, the
    kernel on `stream`, the device->host copies on a third, ordered by events
    so that step i's inputs land while step i-1 computes and step i-2's
    outputs drain. Every step's copies are inside the timed region."""
    from exact_attention_54_gb300.metrics import attention_flops, decode_bytes
    n = max(1, min(args.e2e_steps, args.steps))
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    S = wd.num_splits

    def buffers(kind):
        if kind == "prefill":
            host_in = [t.cpu().pin_memory() for t in pre]
            sets = []
            for _ in range(2):
                q, k, v = (torch.empty_like(t, device=dev) for t in pre)
                sets.append({"in": (q, k, v), "o": torch.empty_like(q),
                             "lse": torch.empty(wp.B, wp.H, wp.Sq, dtype=torch.float32, device=dev),
                             "ho": torch.empty(wp.B, wp.H, wp.Sq, wp.D, dtype=wp.dtype).pin_memory(),
                             "hl": torch.empty(wp.B, wp.H, wp.Sq, dtype=torch.float32).pin_memory()})
            return host_in, sets
        host_in = [t.cpu().pin_memory() for t in dec]
        sets = []
        for _ in range(2):
            q, k, v = (torch.empty_like(t, device=dev) for t in dec)
            sets.append({"in": (q, k, v),
                         "ws": (torch.empty(wd.B, wd.H, S, wd.D, dtype=torch.float32, device=dev),
                                torch.empty(wd.B, wd.H, S, dtype=torch.float32, device=dev),
                                torch.empty(wd.B, wd.H, S, dtype=torch.float32, device=dev)),
                         "counters": torch.zeros(wd.B * wd.H, dtype=torch.int32, device=dev),
                         "o": torch.empty(wd.B, wd.H, 1, wd.D, dtype=wd.dtype, device=dev),
                         "lse": torch.empty(wd.B, wd.H, dtype=torch.float32, device=dev),
                         "ho": torch.empty(wd.B, wd.H, 1, wd.D, dtype=wd.dtype).pin_memory(),
                         "hl": torch.empty(wd.B, wd.H, dtype=torch.float32).pin_memory()})
        return host_in, sets

    out = {}
    for name in ("prefill", "decode"):
        host_in, sets = buffers(name)
        ev = [{k: torch.cuda.Event() for k in ("in", "run", "out")} for _ in range(2)]
        started = [False, False]

        def step(i):
            b, e = sets[i % 2], ev[i % 2]
            with torch.cuda.stream(s_in):
                if started[i % 2]:
                    s_in.wait_event(e["run"])  # the previous kernel on this set has read its inputs
                for d, h in zip(b["in"], host_in):
                    d.copy_(h, non_blocking=True)
                e["in"].record(s_in)
            stream.wait_event(e["in"])
            if started[i % 2]:
                stream.wait_event(e["out"])  # the previous read-back of this set's outputs is done
            q, k, v = b["in"]
            if name == "prefill":
                fa.fa_fwd(q, k, v, b["o"], b["lse"], wp.causal, wp.scale, stream)
            else:
                fa.fa_decode_splitkv_fused(q, k, v, b["o"], b["lse"], *b["ws"], b["counters"], S, wd.scale, stream)
            e["run"].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(e["run"])
                b["ho"].copy_(b["o"], non_blocking=True)
                b["hl"].copy_(b["lse"], non_blocking=True)
                e["out"].record(s_out)
            started[i % 2] = True

        for i in range(2):
            step(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(n):
            step(i)
        torch.cuda.synchronize()
        dt = aggregate_max([time.perf_counter() - t0], world)[0]
        fa.fa_check_device_error()
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sets[0]["ho"].numel() * sets[0]["ho"].element_size() + sets[0]["hl"].numel() * sets[0]["hl"].element_size()
        if name == "prefill":
            val = world * attention_flops(wp.B, wp.H, wp.Sq, wp.Sk, wp.D, wp.causal) * n / dt / 1e12
            unit = "TFLOPS"
        else:
            val = world * decode_bytes(wd.B, wd.H, wd.Sk, wd.D) * n / dt / 1e9
            unit = "GB/s"
        out[name] = {"value": val, "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                     "steps": n, "ms_per_step": 1e3 * dt / n, "copy_gbs": (h2d + d2h) * n / dt / 1e9,
                     "pipelined": "inputs of step i land while step i-1 computes; outputs drain on a third stream"}
        del sets, host_in
    return out


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        backend = "gloo" if args.impl == "reference" else "nccl"
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            line = run_reference(args, rank, world)
        else:
            line = run_gpu(args, rank, world, local)
            if rank == 0 and line is not None and not args.no_cpu_baseline:
                from exact_attention_54_gb300 import inputs
                r, threads, desc, dt = oracle_rate(inputs.WORKLOADS[PREFILL], args.cpu_seconds)
                line["cpu_baseline"] = {"value": r, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
                                        "sample": desc, "seconds": dt}
                r1, t1, desc1, dt1 = oracle_rate(inputs.WORKLOADS[PREFILL], args.cpu_seconds / 3, threads=1)
                line["cpu_baseline"]["single_core"] = {"value": r1, "unit": "TFLOPS", "cores": t1,
                                                       "sample": desc1, "seconds": dt1}
                r2, t2, desc2, dt2 = oracle_decode_rate(inputs.WORKLOADS[DECODE], args.cpu_seconds / 3)
                line["decode"]["cpu_baseline"] = {"value": r2, "unit": "GB/s", "cores": t2, "kind": "oracle",
                                                  "sample": desc2, "seconds": dt2}
        if rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
