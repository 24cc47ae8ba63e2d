#!/usr/bin/env python3
"""Benchmark of the GB300 attention forward: one JSON line on rank 0.

A step is one attention forward over the whole workload (every row of every
head), inputs already resident in HBM.  The default workload is the long,
non-causal, D=128 shape [B=4, H=32, N=16384, D=128] with Q, K ~ N(0, 3^2);
``--workload`` picks another of ``synth.WORKLOADS``.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (torchrun, one rank per GPU): every rank runs the same workload on
its own GPU; (b, h) problems are independent, so there is no data-path
collective and the scaling is weak.  Timing takes the max over ranks.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from attention_forward_12_gb300 import multirank, synth  # noqa: E402

METRIC = "attention fwd TFLOP/s and µs/call at 1 GB300; % of dense FP16 tensor peak"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "peaked_4x32x16384x128"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAK_TFLOPS = 1900.0  # dense bf16 burst, used only without a measured-peaks file


def flops(w: synth.Workload) -> float:
    """4*B*H*Nq*Nk*D, halved when causal (two matmuls of 2*N*N*D each)."""
    f = 4.0 * w.B * w.H * w.Nq * w.Nk * w.D
    return f / 2 if w.causal else f


def algorithmic_bytes(w: synth.Workload) -> int:
    """Q, K, V read once, O and LSE written once."""
    return 2 * w.B * w.H * (w.Nq * w.D * 2 + w.Nk * w.D * 2) + 4 * w.B * w.H * w.Nq


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return None, "fallback"


def gpu_local_cpus(dev_index: int):
    """The CPUs attached to the GPU's PCI root (sysfs local_cpulist), among
    those this process may use; None when unknown.  On a Grace host the
    pinned buffers of the end-to-end leg are first touched from these CPUs,
    so that they sit in the memory of the GPU's own socket."""
    import torch
    p = torch.cuda.get_device_properties(dev_index)
    ids = [getattr(p, a, None) for a in ("pci_domain_id", "pci_bus_id", "pci_device_id")]
    if None in ids:
        return None
    dom, bus, dev = ids
    for d in (f"{dom:04x}", f"{dom:08x}"):
        path = f"/sys/bus/pci/devices/{d}:{bus:02x}:{dev:02x}.0/local_cpulist"
        if not os.path.exists(path):
            continue
        cpus = set()
        for part in open(path).read().strip().split(","):
            if part:
                lo, _, hi = part.partition("-")
                cpus.update(range(int(lo), int(hi or lo) + 1))
        cpus &= os.sched_getaffinity(0)
        return cpus or None
    return None


def _strip_comments(src: str) -> str:
    """C/C++ source without comments, blank lines and the indentation of each
    line (string literals in these files hold no comment markers)."""
    import re
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.strip() for line in src.splitlines() if line.strip())


def kernel_source_digest() -> str:
    """Digest of the kernel source's code (comments do not count), which
    keys the recorded ncu traffic to the code it was measured on."""
    h = hashlib.sha256()
    for rel in ("attention_forward_12_gb300/csrc/attn_fwd.cu",
                "attention_forward_12_gb300/csrc/sm103_primitives.cuh"):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None, None
    with open(p) as f:
        rec = json.load(f)
    ent = rec.get(workload)
    if not ent or ent.get("kernel_digest") != kernel_source_digest():
        return None, None
    return ent.get("dram_bytes_per_launch"), ent.get("note")


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons = [], [], set()
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                clk, cmax = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            sm.append(clk)
            mx.append(cmax)
            names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def oracle_sample(w, q, k, v, seconds: float, seed: int):
    """Time the fp64 oracle on a bounded row sample (~`seconds` of CPU work).

    The sample is made of blocks of 256 random query rows, each block from a
    random (b, h) head, so that the per-row cost includes the oracle's
    per-head set-up in the same proportion as a run over whole heads would.
    One block calibrates the size.  Returns (rows, O, LSE, elapsed, threads,
    flops_done).
    """
    import numpy as np
    import oracle
    gen = np.random.Generator(np.random.Philox(key=[seed, 1234]))
    heads = w.B * w.H
    per_head = min(256, w.Nq)

    def block(h):
        return h * w.Nq + np.sort(gen.choice(w.Nq, size=per_head, replace=False))

    t0 = time.perf_counter()
    oracle.attn_rows(q, k, v, w.scale, w.causal, block(int(gen.integers(heads))))
    dt = max(time.perf_counter() - t0, 1e-4)
    nblocks = max(1.0, seconds / dt)
    if nblocks <= heads:
        hs = np.sort(gen.choice(heads, size=int(nblocks), replace=False))
        rows = np.concatenate([block(int(h)) for h in hs])
    else:  # every head, more rows from each
        per = int(min(w.Nq, per_head * nblocks / heads))
        rows = np.concatenate([h * w.Nq + np.sort(gen.choice(w.Nq, size=per, replace=False))
                               for h in range(heads)])
    t0 = time.perf_counter()
    O, L, threads = oracle.attn_rows(q, k, v, w.scale, w.causal, rows)
    el = time.perf_counter() - t0
    i = rows % w.Nq
    keys = np.minimum(i + 1, w.Nk) if w.causal else np.full(rows.shape, w.Nk)
    done = float(np.sum(4.0 * keys.astype(np.float64) * w.D))  # exact flops of the sampled rows
    return rows, O, L, el, threads, done


def run_reference(args, w):
    """The reference arm: the fp64 CPU oracle as it stands, on host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    q, k, v = synth.workload_qkv(w)
    total = args.steps + args.warmup
    per_step = max(0.2, min(10.0, 150.0 / max(total, 1)))
    times, rates = [], []
    threads = 0
    nrows = 0
    for s in range(total):
        rows, _, _, el, threads, done = oracle_sample(w, q, k, v, per_step, seed=w.seed + s)
        if s >= args.warmup:
            times.append(el)
            rates.append(done / el / 1e12)
            nrows = len(rows)
    value = statistics.median(rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.median(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{nrows} query rows per step, in blocks of random rows of "
                                   f"random heads of the workload (~{per_step:.1f} s of CPU work each)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def percentile(xs, pct):
    """Linear-interpolated percentile of a non-empty list (numpy's default rule)."""
    ys = sorted(xs)
    x = (len(ys) - 1) * pct / 100.0
    lo = int(x)
    hi = min(lo + 1, len(ys) - 1)
    return ys[lo] + (ys[hi] - ys[lo]) * (x - lo)


def config_of(w, splits=0):
    return {"workload": w.name, "split_kv_shares": splits, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "D": w.D,
            "causal": w.causal, "scale": w.scale, "sigma_qk": w.sigma_qk, "sigma_v": w.sigma_v,
            "seed": w.seed,
            "l2": ("inputs larger than L2 (%.0f MB > 129 MB); no flush" % (algorithmic_bytes(w) / 1e6))
            if algorithmic_bytes(w) > L2_BYTES else "L2 flushed between steps (256 MB write)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--shape", default=None,
                    help="B,H,N,D,causal or B,H,Nq,Nk,D,causal: a custom N(0,1) workload "
                         "instead of --workload (small profiling captures, decode shapes)")
    ap.add_argument("--splits", type=int, default=0,
                    help="time the split-KV forward with this many key shares (-1: the "
                         "library's suggestion; 0: the single-pass forward)")
    ap.add_argument("--dtype", choices=["f16", "e4m3"], default="f16",
                    help="input precision: fp16 (attn_fwd) or FP8 E4M3 (attn_fwd_fp8, D = 128)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--host-chunks", type=int, default=32,
                    help="head chunks of attn_fwd_host, the end-to-end leg's call (fp16 single pass)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()
    w = synth.WORKLOADS[args.workload]
    if args.shape:
        vals = [int(x) for x in args.shape.split(",")]
        if len(vals) == 5:
            B, H, N, D, c = vals
            Nq = Nk = N
        else:
            B, H, Nq, Nk, D, c = vals
        name = f"custom_{B}x{H}x{Nq}x{D}" if Nq == Nk else f"custom_{B}x{H}x{Nq}x{Nk}x{D}"
        w = synth.Workload(name + ("_causal" if c else ""), B, H, Nq, Nk, D, bool(c), 1.0, 1.0, 42)
    if args.impl == "reference":
        return run_reference(args, w)

    import torch
    import attention_forward_12_gb300 as attn

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    attn.load_library()

    # inputs: seeded on the host (the same bytes the oracle sees), copied once;
    # every rank draws its own independent problems of the workload's shape
    fp8 = args.dtype == "e4m3"
    if fp8 and (w.D != 128 or args.splits != 0):
        raise SystemExit("--dtype e4m3 runs the single-pass forward at D = 128")
    gen_qkv = synth.make_qkv_e4m3 if fp8 else synth.make_qkv
    qn, kn, vn = gen_qkv(w.B, w.H, w.Nq, w.Nk, w.D, multirank.rank_seed(w.seed, rank), w.sigma_qk, w.sigma_v)
    q = torch.from_numpy(qn).to(dev)
    k = torch.from_numpy(kn).to(dev)
    v = torch.from_numpy(vn).to(dev)
    o = torch.empty((w.B, w.H, w.Nq, w.D), dtype=torch.float16, device=dev)
    lse = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    flush = None
    if algorithmic_bytes(w) <= L2_BYTES:
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    splits = args.splits
    if splits < 0:
        splits = max(1, attn.splitkv_suggest(w.B, w.H, w.Nq, w.Nk, w.D, w.causal))
    ws = None
    if splits > 0:  # workspace allocated once, outside every timed region
        ws_bytes = attn.splitkv_workspace_bytes(w.B, w.H, w.Nq, w.D, splits)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    if fp8:  # V^T workspace, allocated once outside every timed region
        ws_bytes = attn.fp8_workspace_bytes(w.B, w.H, w.Nk, w.D)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    # kernels per step: the forward and the merge (split-KV), else what the
    # library reports for the single pass, plus the V transpose for E4M3
    if splits > 0:
        launches_per_step = 2
    else:
        launches_per_step = attn.fwd_launch_count(w.B, w.H, w.Nq, w.Nk, w.D, w.causal) + (1 if fp8 else 0)

    def call():
        """One forward through the C ABI on the launching stream."""
        if fp8:
            code = attn.attn_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                     w.B, w.H, w.Nq, w.Nk, w.D, w.scale, w.causal, 1.0, 1.0, 1.0,
                                     ws.data_ptr(), ws.numel(), sptr)
        elif splits > 0:
            code = attn.attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), w.B, w.H, w.Nq, w.Nk, w.D, w.scale, w.causal,
                                         splits, ws.data_ptr(), ws.numel(), sptr)
        else:
            code = attn.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                 w.B, w.H, w.Nq, w.Nk, w.D, w.scale, w.causal, sptr)
        if code != attn.ATTN_OK:
            raise attn.AttnError(code, "attn_fwd")

    def step():
        if flush is not None:
            flush.fill_(1)
        call()

    def barrier():
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    barrier()
    if attn.get_status(sptr) != attn.ATTN_OK:
        raise RuntimeError("kernel status error during warm-up")

    # ---------------- device-timed region: K steps, inputs resident
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        barrier()
        t_start.record(stream)
        for s in range(args.steps):
            if flush is not None:
                flush.fill_(1)
            ev[s][0].record(stream)
            call()
            ev[s][1].record(stream)
        t_end.record(stream)
        barrier()
    status = attn.get_status(sptr)
    if status != attn.ATTN_OK:
        raise RuntimeError(f"kernel status {status} in the timed region")
    kernel_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = t_start.elapsed_time(t_end)
    if flush is not None:
        step_ms = statistics.mean(kernel_ms)
    else:
        step_ms = total_ms / args.steps
    step_ms = multirank.max_over_ranks(step_ms, dist, dev)
    f = flops(w)
    value = multirank.aggregate_tflops(f, world, step_ms)
    kern_avg_ms = statistics.mean(kernel_ms)

    # ---------------- end to end: host buffers, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        saved_affinity = os.sched_getaffinity(0)
        local_cpus = gpu_local_cpus(local_rank)
        if local_cpus:  # first touch of the pinned pages on the GPU's own socket
            os.sched_setaffinity(0, local_cpus)
        try:
            hq, hk, hv = (torch.from_numpy(x).pin_memory() for x in (qn, kn, vn))
            ho = torch.empty(o.shape, dtype=torch.float16).pin_memory()
            hl = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
            ho.zero_()
            hl.zero_()
        finally:
            os.sched_setaffinity(0, saved_affinity)

        host_entry = splits == 0

        def e2e_step():
            # the library's host-buffer entries: copies overlapped with the forward
            if host_entry and fp8:
                code = attn.attn_fwd_fp8_host(hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), ho.data_ptr(),
                                              hl.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                              lse.data_ptr(), w.B, w.H, w.Nq, w.Nk, w.D, w.scale, w.causal,
                                              1.0, 1.0, 1.0, ws.data_ptr(), ws.numel(), args.host_chunks, sptr)
                if code != attn.ATTN_OK:
                    raise attn.AttnError(code, "attn_fwd_fp8_host")
                return
            if host_entry:
                code = attn.attn_fwd_host(hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), ho.data_ptr(), hl.data_ptr(),
                                          q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                          w.B, w.H, w.Nq, w.Nk, w.D, w.scale, w.causal, args.host_chunks, sptr)
                if code != attn.ATTN_OK:
                    raise attn.AttnError(code, "attn_fwd_host")
                return
            q.copy_(hq, non_blocking=True)
            k.copy_(hk, non_blocking=True)
            v.copy_(hv, non_blocking=True)
            call()
            ho.copy_(o, non_blocking=True)
            hl.copy_(lse, non_blocking=True)

        # The box's pinned host-to-device and device-to-host bandwidths, for
        # reading the end-to-end figure: the forward hides its copies only
        # while they run faster than it consumes and produces the data.
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        q.copy_(hq, non_blocking=True)
        a.record(stream)
        q.copy_(hq, non_blocking=True)
        b.record(stream)
        b.synchronize()
        h2d_gbs = hq.numel() * hq.element_size() / (a.elapsed_time(b) * 1e-3) / 1e9
        a.record(stream)
        ho.copy_(o, non_blocking=True)
        b.record(stream)
        b.synchronize()
        d2h_gbs = ho.numel() * ho.element_size() / (a.elapsed_time(b) * 1e-3) / 1e9
        n_e2e = max(3, min(args.steps, 10))
        for _ in range(2):
            e2e_step()
        barrier()
        # one event per step boundary on the caller's stream (each call's
        # copies and forward start after the previous call's last copy out)
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e + 1)]
        marks[0].record(stream)
        for s in range(n_e2e):
            e2e_step()
            marks[s + 1].record(stream)
        barrier()
        step_e2e = [marks[s].elapsed_time(marks[s + 1]) for s in range(n_e2e)]
        e_ms = marks[0].elapsed_time(marks[n_e2e]) / n_e2e
        e_ms = multirank.max_over_ranks(e_ms, dist, dev)
        e2e = {"value": multirank.aggregate_tflops(f, world, e_ms), "unit": UNIT, "ms_per_step": e_ms,
               "steps": n_e2e,
               "step_ms": {"median": statistics.median(step_e2e), "p10": percentile(step_e2e, 10),
                           "p90": percentile(step_e2e, 90), "max": max(step_e2e)},
               "h2d_gbs_measured": h2d_gbs,
               "d2h_gbs_measured": d2h_gbs,
               "host_buffers": (f"pinned, first touched on the {len(local_cpus)} CPUs local to the GPU"
                                if local_cpus else "pinned (GPU-local CPUs unknown)"),
               "call": (f"{'attn_fwd_fp8_host' if fp8 else 'attn_fwd_host'}, {args.host_chunks} head chunks, "
                        f"pinned host buffers" if host_entry
                        else "copies in, forward, copies out on one stream, pinned host buffers"),
               "h2d_bytes_per_step": int(hq.numel() * hq.element_size() + hk.numel() * hk.element_size()
                                         + hv.numel() * hv.element_size()),
               "d2h_bytes_per_step": int(ho.numel() * 2 + hl.numel() * 4)}
        assert attn.get_status(sptr) == attn.ATTN_OK

    if rank != 0:
        if dist is not None:
            dist.barrier()
            dist.destroy_process_group()
        return 0

    peaks, peak_src = read_peaks()
    if peaks:
        peak = float(peaks["bf16_tflops"])  # fp16 dense rate = bf16 dense rate (nominal 1:1)
        peak_sus = float(peaks.get("bf16_tflops_sustained", peak))
    else:
        peak = peak_sus = FALLBACK_PEAK_TFLOPS
    peak_note = f"bf16_tflops (burst) of {peak_src}; fp16 dense = bf16 dense"
    nominal = 2250.0
    if fp8:  # no measured fp8 peak: the bf16 one times the nominal dense ratio 4.5 / 2.25
        peak, peak_sus, nominal = 2.0 * peak, 2.0 * peak_sus, 4500.0
        peak_note = f"2 x bf16_tflops (burst) of {peak_src}: fp8 dense = 2 x bf16 dense nominally"
    achieved = f / (kern_avg_ms * 1e-3) / 1e12
    traffic, traffic_note = recorded_traffic(w.name + ("_e4m3" if fp8 else ""))
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": peak_note,
                "peak_sustained": peak_sus, "frac_sustained": achieved / peak_sus,
                f"frac_of_nominal_{int(nominal)}": achieved / nominal,
                "kernel_ms_avg": kern_avg_ms, "kernel_ms_min": min(kernel_ms),
                "algorithmic_flops_per_launch": f}
    if traffic_note:
        roofline["traffic_note"] = traffic_note

    cpu = None
    if world == 1:
        import numpy as np
        if fp8:  # the oracle on the exactly decoded inputs (every E4M3 value is an fp16 value)
            import oracle
            qo, ko, vo = (oracle.e4m3_to_double(x).astype(np.float16) for x in (qn, kn, vn))
        else:
            qo, ko, vo = qn, kn, vn
        rows, O, L, el, threads, done = oracle_sample(w, qo, ko, vo, args.cpu_seconds, seed=w.seed)
        og = o.view(-1, w.D)[torch.from_numpy(rows).to(dev)].float().cpu().numpy().astype(np.float64)
        lg = lse.view(-1)[torch.from_numpy(rows).to(dev)].cpu().numpy().astype(np.float64)
        cpu = {"value": done / el / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{len(rows)} query rows of the same workload, in blocks of random "
                         f"rows of random heads (fp64 oracle, {el:.1f} s)",
               "gpu_vs_oracle_on_sample": {"o_max_abs": float(np.abs(og - O).max()),
                                           "o_rel_rms": float(np.linalg.norm(og - O) / np.linalg.norm(O)),
                                           "lse_max_abs": float(np.abs(lg - L).max())}}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "us_per_call": step_ms * 1e3,
        "pct_of_peak": 100.0 * value / world / peak,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.dtype,
        "data": "synthetic", "config": config_of(w, splits), "parallelism": f"replicas x{world} (independent problems)",
        "gpu_launches": args.steps * launches_per_step, "roofline": roofline, "clocks": clk.summary(),
        "e2e": e2e, "cpu_baseline": cpu,
        # per-call device time of this rank: each step's own pair of events
        "call_us": {"median": 1e3 * statistics.median(kernel_ms), "p10": 1e3 * percentile(kernel_ms, 10),
                    "p90": 1e3 * percentile(kernel_ms, 90), "n": len(kernel_ms)},
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
