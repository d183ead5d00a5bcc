#!/usr/bin/env python
"""Throughput benchmark of the fused attention hot path on GB300.

One step = one full pass of the path over the long-context causal workload
(b=1, h=32, s=16384, d=128, bf16, Q and K scaled by 2): the forward kernel
(O and LSE) followed by the backward chain (preprocess, main, dQ convert)
that produces dQ, dK, dV.  FLOPs per step follow the pages' count
4*b*h*s*s*d*0.5 for the causal forward ("Inside NVIDIA's cuDNN Graph API",
section 5) and 2.5x that for the backward (five s x s x d products against
the forward's two), 3.5x in total.

The K timed steps give the line's value (CUDA events around each step only,
an L2 flush before each); K more steps with events around the forward kernel
and the backward's main kernel give the per-kernel phases and the roofline.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Prints one JSON line on rank 0.  For N > 1 each rank runs an independent
replica of the workload on its own GPU (the path has no cross-GPU exchange),
so the scaling is weak; the time is the maximum over ranks.

``--impl reference`` times the fp64 CPU oracle on the host cores instead, on
a bounded sample of the same workload (rank 0 only).

``--variant`` measures the widened rows on the same workload (the headline
line is the default, bf16): ``deterministic`` runs the backward with its
deterministic dQ pass (the backward timer then spans the main kernel and the
dQ pass), ``fp8`` times the E4M3 forward alone (bf16 output) against the FP8
tensor peak (the measured bf16 peak x 2, the nominal FP8/BF16 ratio).  The
mask and head-sharing rows run the forward + backward step through the
extended calls: ``gqa`` with 8 key/value heads for the 32 query heads,
``window`` with the causal mask and window_left = 2048, ``bottom_right`` with
4096 queries against the 16384 keys under the bottom-right causal mask.  Their
FLOPs count the visible (query, key) pairs exactly (4*d per pair forward,
2.5x that backward), since the pages' halving applies to the plain causal
square only.
"""
from __future__ import annotations

import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "SDPA fwd/bwd TFLOP/s (causal-halved FLOPs), % of GB300 BF16 tensor peak"
WORKLOAD = "c5_b1h32s16384d128_causal_qk2"
BWD_FACTOR = 2.5          # backward FLOPs per forward FLOP
L2_FLUSH_BYTES = 512 << 20  # > 2x the 129 MB L2
REF_PREFIX = 2048         # tokens of one head per oracle sample

# DRAM bytes per launch of the dominant kernel from one ncu capture of the
# full workload (dram__bytes_read.sum + dram__bytes_write.sum), keyed by kernel
# and the library version the capture was taken with; any other version
# reports null.  Source: profiles/bwd_main_dram_c5_b1h32s16384d128.md.
TRAFFIC = {("bwd_main", "sdpa_gb300 0.4 sm_103a"): 0.81430e9 + 0.49046e9,
           ("bwd_main", "sdpa_gb300 0.6 sm_103a"): 0.83157e9 + 0.50512e9,
           # bwd.cu is unchanged from 0.6 to 0.10 (only the forwards changed)
           ("bwd_main", "sdpa_gb300 0.7 sm_103a"): 0.83157e9 + 0.50512e9,
           ("bwd_main", "sdpa_gb300 0.8 sm_103a"): 0.83157e9 + 0.50512e9,
           ("bwd_main", "sdpa_gb300 0.9 sm_103a"): 0.83157e9 + 0.50512e9,
           ("bwd_main", "sdpa_gb300 0.10 sm_103a"): 0.83157e9 + 0.50512e9,
           # 0.11 changed the CTA order of small and packed problems only
           ("bwd_main", "sdpa_gb300 0.11 sm_103a"): 0.832530e9 + 0.505720e9,
           # 0.12: programmatic dependent launch across the backward chain
           ("bwd_main", "sdpa_gb300 0.12 sm_103a"): 0.831935e9 + 0.505143e9,
           ("bwd_main", "sdpa_gb300 0.13 sm_103a"): 0.831402e9 + 0.505376e9,
           # 0.14: dK, dV written as whole 128-byte lines (staged in shared memory)
           ("bwd_main", "sdpa_gb300 0.14 sm_103a"): 0.84556e9 + 0.51496e9,
           # 0.15 changed the forwards' O stores only
           ("bwd_main", "sdpa_gb300 0.15 sm_103a"): 0.84556e9 + 0.51496e9,
           # 0.16 changed the two-tile forward's list of non-causal dense problems only
           ("bwd_main", "sdpa_gb300 0.16 sm_103a"): 0.84556e9 + 0.51496e9,
           # 0.17 changed the one-tile forward's packed schedule only
           ("bwd_main", "sdpa_gb300 0.17 sm_103a"): 0.84556e9 + 0.51496e9,
           # 0.18 changed the two-tile forward's packed schedule and the forward choice only
           ("bwd_main", "sdpa_gb300 0.18 sm_103a"): 0.84556e9 + 0.51496e9,
           # 0.19 and 0.20 changed the two-tile forward's load barriers only
           ("bwd_main", "sdpa_gb300 0.19 sm_103a"): 0.84556e9 + 0.51496e9,
           ("bwd_main", "sdpa_gb300 0.20 sm_103a"): 0.84556e9 + 0.51496e9,
           # 0.21 changed the one-tile forward's load barriers only
           ("bwd_main", "sdpa_gb300 0.21 sm_103a"): 0.84556e9 + 0.51496e9,
           # 0.22 changed the deterministic dQ pass only
           ("bwd_main", "sdpa_gb300 0.22 sm_103a"): 0.84556e9 + 0.51496e9,
           # 0.23: two of bwd_main's barriers folded into others; captured again
           ("bwd_main", "sdpa_gb300 0.23 sm_103a"): 0.84483e9 + 0.51597e9,
           # 0.24 changed the one-tile forward only
           ("bwd_main", "sdpa_gb300 0.24 sm_103a"): 0.84483e9 + 0.51597e9}


def fwd_flops(w) -> float:
    return 4.0 * w.b * w.h * w.s * w.s * w.d * (0.5 if w.causal else 1.0)


# Extended-call variants on the default workload: key/value heads, query
# length, mask (0 none, 1 top-left causal, 2 bottom-right causal), window_left.
EXT_VARIANTS = {"gqa": dict(h_kv=8, s_q=None, mask=1, window=-1),
                "window": dict(h_kv=None, s_q=None, mask=1, window=2048),
                "bottom_right": dict(h_kv=None, s_q=4096, mask=2, window=-1)}


def visible_pairs(s_q: int, s_kv: int, mask: int, window: int) -> int:
    """(query, key) pairs the mask leaves visible in one (b, h) slice: row i
    sees keys [max(0, i + delta - window), min(s_kv, i + delta + 1)) with
    delta = s_kv - s_q for the bottom-right mask and 0 otherwise (no upper
    bound without a causal mask, no lower bound without a window)."""
    import numpy as np
    i = np.arange(s_q, dtype=np.int64)
    delta = s_kv - s_q if mask == 2 else 0
    hi = np.minimum(s_kv, i + delta + 1) if mask != 0 else np.full(s_q, s_kv, np.int64)
    lo = np.maximum(0, i + delta - window) if window >= 0 else np.zeros(s_q, np.int64)
    return int(np.maximum(hi - lo, 0).sum())


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="dense workload name from sdpa_inputs.WORKLOADS (profiling runs); the "
                         "reported metric is quoted on the default")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle CPU-baseline leg")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--configs", action="store_true",
                    help="instead of the benchmark line: time the forward and the backward "
                         "chain of every configured workload, one JSON line each")
    ap.add_argument("--only", default=None, help="with --configs: this workload only")
    ap.add_argument("--probe", action="store_true",
                    help="with --configs --only: run the forward and backward three times "
                         "and print nothing else (a launch set for a profiler)")
    ap.add_argument("--variant", choices=["bf16", "deterministic", "fp8"] + list(EXT_VARIANTS),
                    default="bf16",
                    help="bf16 (default, the headline), deterministic backward, FP8 forward, or "
                         "an extended-call row (gqa, window, bottom_right)")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest x over all ranks: the job takes as long as its slowest rank."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(flops_per_step: float, steps: int, world: int, max_total_ms: float) -> float:
    """Whole-job TFLOP/s: the steps of every rank (each a full replica of the
    workload) over the slowest rank's time, i.e. weak scaling."""
    return world * flops_per_step * steps / (max_total_ms * 1e-3) / 1e12


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


class ClockSampler:
    """nvidia-smi sampled every 100 ms during the timed region."""

    FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.lines: list[str] = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.5)  # let the first samples arrive before the timed region

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        rows = []
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 10:
                continue
            if self.uuid and parts[1] != self.uuid:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1] or rows
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({name for r in inside for name, v in zip(self.REASONS, r[3])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside)}


# ---------------------------------------------------------------------- oracle legs
def oracle_sample_rate(w, t, min_s: float, max_s: float, heads=None):
    """Time the fp64 oracle (fwd + bwd) on causal prefixes of single heads.

    Each sample is head h of the workload's own inputs cut to its first
    REF_PREFIX tokens, a self-contained causal problem with the same
    arithmetic per score.  Returns (TFLOP/s, seconds, samples, threads).
    """
    import oracle
    L = min(REF_PREFIX, w.s)
    flops = 4.0 * L * L * w.d * 0.5 * (1.0 + BWD_FACTOR)
    done, spent, h = 0, 0.0, 0
    order = heads if heads is not None else range(10 ** 9)
    for h in order:
        hh = h % w.h
        q = t["q"][0:1, hh:hh + 1, :L]
        k = t["k"][0:1, hh:hh + 1, :L]
        v = t["v"][0:1, hh:hh + 1, :L]
        do = t["do"][0:1, hh:hh + 1, :L]
        t0 = time.perf_counter()
        oracle.sdpa_fwd(q, k, v, w.scale, w.causal)
        oracle.sdpa_bwd(q, k, v, do, w.scale, w.causal)
        spent += time.perf_counter() - t0
        done += 1
        if heads is None and (spent >= min_s or spent + spent / done > max_s):
            break
    return flops * done / spent / 1e12, spent, done, oracle.num_threads()


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import sdpa_inputs
    import oracle
    oracle.build()
    w = sdpa_inputs.WORKLOADS[args.workload]
    t = sdpa_inputs.make(w)
    oracle_sample_rate(w, t, 0, 0, heads=range(args.warmup))
    rate, spent, n, threads = oracle_sample_rate(w, t, 0, 0, heads=range(args.steps))
    L = min(REF_PREFIX, w.s)
    sample = (f"per step: one head of {w.name} (heads in turn) cut to its first {L} tokens, "
              f"causal fp64 forward + backward")
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": spent / n * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample_prefix_tokens": L},
        "cpu_baseline": {"value": rate, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": rate, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------- our arm
def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import sdpa_inputs
    import scaled_dot_product_04_gb300 as sdpa
    sdpa.load()

    w = sdpa_inputs.WORKLOADS[args.workload]
    if w.layout != "bhsd":
        raise SystemExit(f"bench.py times dense workloads; {w.name} is packed")
    t = sdpa_inputs.make(w)
    b, h, s, d = w.b, w.h, w.s, w.d
    scale, causal = w.scale, int(w.causal)
    variant = args.variant
    fp8 = variant == "fp8"
    det = 1 if variant == "deterministic" else 0
    ext = EXT_VARIANTS.get(variant)
    hk, s_q, mask, window = h, s, causal, -1
    if ext:
        hk = ext["h_kv"] or h
        s_q = ext["s_q"] or s
        mask, window = ext["mask"], ext["window"]
        qq, kk, vv, dd = sdpa_inputs.dense(b, h, s_q, s, d, w.seed, qk_mult=w.qk_mult, h_kv=hk)
        t = dict(t, q=qq, k=kk, v=vv, do=dd)
    if fp8:
        # E4M3 codes of the workload's own Q, K, V with per-tensor descales
        enc = [sdpa_inputs.fp8_quantize(t[x].float()) for x in ("q", "k", "v")]
        t = dict(t, q=enc[0][0], k=enc[1][0], v=enc[2][0])
        descales = [torch.tensor([e[1]], dtype=torch.float32, device=dev) for e in enc]
    q, k, v, do = (t[x].to(dev) for x in ("q", "k", "v", "do"))
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty((b, h, s_q), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(do), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(max(1, sdpa.sdpa_bwd_ex_workspace_size(b, h, s_q, d, det)),
                     dtype=torch.uint8, device=dev)
    amax = torch.empty(1, dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    f_fwd = 4.0 * b * h * d * visible_pairs(s_q, s, mask, window) if ext else fwd_flops(w)
    f_step = f_fwd if fp8 else f_fwd * (1.0 + BWD_FACTOR)

    def step(ev_f=None, ev_b=None):
        if ev_f:
            sdpa.sdpa_set_kernel_timer(*ev_f)
        if fp8:
            sdpa.sdpa_fwd_fp8(q, k, v, o, lse, *descales, None, amax, b, h, h, s, s, d, scale,
                              causal, -1, 0, stream)
            sdpa.sdpa_set_kernel_timer(None, None)
            return
        if ext:
            sdpa.sdpa_fwd_ex(q, k, v, o, lse, b, h, hk, s_q, s, d, scale, mask, window, 0, stream)
        else:
            sdpa.sdpa_fwd(q, k, v, o, lse, b, h, s, s, d, scale, causal, 0, stream)
        if ev_b:
            sdpa.sdpa_set_kernel_timer(*ev_b)
        if ext:
            sdpa.sdpa_bwd_ex(q, k, v, o, do, lse, dq, dk, dv, b, h, hk, s_q, s, d, scale, mask,
                             window, 0, 0, ws, ws.numel(), stream)
        elif det:
            sdpa.sdpa_bwd_ex(q, k, v, o, do, lse, dq, dk, dv, b, h, h, s, s, d, scale, causal, -1,
                             1, 0, ws, ws.numel(), stream)
        else:
            sdpa.sdpa_bwd(q, k, v, o, do, lse, dq, dk, dv, b, h, s, s, d, scale, causal, 0, ws,
                          ws.numel(), stream)
        sdpa.sdpa_set_kernel_timer(None, None)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    sdpa.sdpa_check_device_error(stream)

    def new_ev():
        return torch.cuda.Event(enable_timing=True)

    # Two timed loops of K steps each, an L2 flush before every step (outside
    # the events).  The first times whole steps only: nothing is recorded
    # between the kernels, so the backward chain's kernels may overlap their
    # neighbours (programmatic dependent launch) as in a caller's own loop; it
    # gives `value`.  The second records the kernel timer's events around the
    # forward kernel and the backward's main kernel; it gives the phases and
    # the roofline of the dominant kernel.
    ev = [(new_ev(), new_ev()) for _ in range(args.steps)]
    evk = [(new_ev(), new_ev(), (new_ev(), new_ev()), (new_ev(), new_ev()))
           for _ in range(args.steps)]
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    for i in range(args.steps):
        flush.zero_()
        evk[i][0].record(stream)
        step(evk[i][2], evk[i][3])
        evk[i][1].record(stream)
    torch.cuda.synchronize(dev)
    t2 = time.time()
    sampler.stop()
    sdpa.sdpa_check_device_error(stream)

    step_ms = [a.elapsed_time(bb) for a, bb in ev]
    kstep_ms = [a.elapsed_time(bb) for a, bb, _, _ in evk]
    fwd_ms = [f[0].elapsed_time(f[1]) for _, _, f, _ in evk]
    bwd_ms = [0.0 if fp8 else g[0].elapsed_time(g[1]) for _, _, _, g in evk]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    value = job_rate(f_step, args.steps, world, total_ms)
    clocks = sampler.summary(t0, t2)

    # ------------------------------------------------------------ end to end
    # Each step copies its inputs from pinned host memory, runs the path and
    # copies its results back.  Three device buffer sets and two copy streams
    # (host->device and device->host, one copy engine each) let step i's
    # copies overlap the compute of its neighbours; every step's own copies
    # stay inside the timed region.  A set is refilled only once its previous
    # results have reached the host, so with two sets a set's result copy,
    # its next input copy and its compute would run back to back: (D2H + H2D
    # + compute) / 2 a step, which a host link sharing its bandwidth between
    # the two directions makes longer than the compute.  Three sets spread
    # that chain over three steps.
    e2e = None
    if not args.no_e2e:
        names_in = ["q", "k", "v"] + ([] if fp8 else ["do"])
        host_in = [t[x].pin_memory() for x in names_in]

        def dev_set():
            ins = [torch.empty(x.shape, dtype=x.dtype, device=dev) for x in host_in]
            outs = [torch.empty_like(o), torch.empty_like(lse)]
            if not fp8:
                outs += [torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv)]
            return ins, outs

        n_sets = 3
        sets = [dev_set() for _ in range(n_sets)]
        host_out = [[torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in sets[0][1]]
                    for _ in range(n_sets)]
        ws_sets = [ws] + [torch.empty_like(ws) for _ in range(n_sets - 1)]
        h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def run_step(i):
            ins, outs = sets[i % n_sets]
            qq, kk, vv = ins[0], ins[1], ins[2]
            oo, ll = outs[0], outs[1]
            if fp8:
                sdpa.sdpa_fwd_fp8(qq, kk, vv, oo, ll, *descales, None, amax, b, h, h, s, s, d,
                                  scale, causal, -1, 0, stream)
                return
            ddo = ins[3]
            gq, gk, gv = outs[2], outs[3], outs[4]
            wsi = ws_sets[i % n_sets]
            if ext:
                sdpa.sdpa_fwd_ex(qq, kk, vv, oo, ll, b, h, hk, s_q, s, d, scale, mask, window, 0,
                                 stream)
                sdpa.sdpa_bwd_ex(qq, kk, vv, oo, ddo, ll, gq, gk, gv, b, h, hk, s_q, s, d, scale,
                                 mask, window, 0, 0, wsi, wsi.numel(), stream)
                return
            sdpa.sdpa_fwd(qq, kk, vv, oo, ll, b, h, s, s, d, scale, causal, 0, stream)
            if det:
                sdpa.sdpa_bwd_ex(qq, kk, vv, oo, ddo, ll, gq, gk, gv, b, h, h, s, s, d, scale,
                                 causal, -1, 1, 0, wsi, wsi.numel(), stream)
            else:
                sdpa.sdpa_bwd(qq, kk, vv, oo, ddo, ll, gq, gk, gv, b, h, s, s, d, scale, causal, 0,
                              wsi, wsi.numel(), stream)

        def pipeline(n):
            free = [None] * n_sets  # device->host copy of the set's last results done
            for i in range(n):
                st = i % n_sets
                ins, outs = sets[st]
                with torch.cuda.stream(h2d):
                    if free[st] is not None:
                        h2d.wait_event(free[st])
                    for dst, src in zip(ins, host_in):
                        dst.copy_(src, non_blocking=True)
                    ready = torch.cuda.Event()
                    ready.record(h2d)
                stream.wait_event(ready)
                run_step(i)
                done = torch.cuda.Event()
                done.record(stream)
                with torch.cuda.stream(d2h):
                    d2h.wait_event(done)
                    for dst, src in zip(host_out[st], outs):
                        dst.copy_(src, non_blocking=True)
                    free[st] = torch.cuda.Event()
                    free[st].record(d2h)

        # the first step's input copy and the last step's result copy cannot
        # overlap any compute; 100 steps (more when more are timed, up to 150)
        # spread that fill and drain thinly, as a caller's long loop would
        n_e2e = max(100, min(args.steps, 150))
        pipeline(n_sets)
        torch.cuda.synchronize(dev)
        ev_a, ev_z = new_ev(), new_ev()
        ev_a.record(h2d)             # before the first step's first copy
        pipeline(n_e2e)
        ev_z.record(d2h)             # after the last step's last copy
        torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(ev_a.elapsed_time(ev_z) / n_e2e, world, dev)
        h2d_bytes = sum(x.numel() * x.element_size() for x in host_in)
        d2h_bytes = sum(x.numel() * x.element_size() for x in host_out[0])
        e2e = {"value": world * f_step / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
               "ms_per_step": e_ms, "steps": n_e2e,
               "copies": "pinned host buffers; three device buffer sets and two copy streams "
                         "overlap each step's copies with the neighbouring steps' compute; "
                         "CUDA events before the first copy and after the last (the "
                         "pipeline's fill and drain included)"}

    # ------------------------------------------------------------ roofline
    # Per-kernel figures use the median over the timed steps (an L2 flush
    # precedes every step).  The denominator is the measured burst peak while
    # the timed region lasts under two seconds (the clocks sampled above stay
    # near the maximum then), else the sustained peak measured under the
    # power cap over seconds.
    peaks, peak_src = read_peaks()
    med_f, med_b = statistics.median(fwd_ms), statistics.median(bwd_ms)
    med_step = statistics.median(step_ms)
    kern = "bwd_main" if sum(bwd_ms) >= sum(fwd_ms) else "fwd"
    if det and kern == "bwd_main":
        kern = "bwd_main+dq"
    k_flops = f_fwd * BWD_FACTOR if kern.startswith("bwd") else f_fwd
    k_ms = med_b if kern.startswith("bwd") else med_f
    achieved = k_flops / (k_ms * 1e-3) / 1e12
    ratio = 2.0 if fp8 else 1.0  # nominal FP8 / BF16 dense tensor rate
    timed_s = (sum(step_ms) + sum(kstep_ms)) * 1e-3
    sustained = timed_s >= 2.0
    burst = float(peaks["bf16_tflops"]) * ratio
    peak = float(peaks["bf16_tflops_sustained"]) * ratio if sustained else burst
    version = sdpa.sdpa_version()
    # the captures are of the default workload and variant
    tr = TRAFFIC.get((kern, version)) if variant == "bf16" and w.name == WORKLOAD else None
    src = ("measured " if peak_src == "measured" else "fallback ") + \
        ("sustained" if sustained else "burst") + " bf16" + \
        (" (MEASURED_PEAKS.json)" if peak_src == "measured" else "") + \
        f", timed region {timed_s:.2f} s" + (" x 2 (nominal FP8/BF16 ratio)" if fp8 else "")
    hbm = float(peaks["hbm_gbs"])
    dram_gbs = tr / (k_ms * 1e-3) / 1e9 if tr else None
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": tr, "kernel": kern, "peak_source": src,
                "kernel_ms_median": k_ms,
                "dram_gbs": dram_gbs, "dram_frac": dram_gbs / hbm if dram_gbs else None,
                "hbm_peak_gbs": hbm}

    def rate(flops, ms):
        return flops / (ms * 1e-3) / 1e12

    phases = {
        "fwd_kernel": {"ms_median": med_f, "ms_mean": statistics.mean(fwd_ms),
                       "tflops": rate(f_fwd, med_f), "frac_burst": rate(f_fwd, med_f) / burst,
                       "frac_sustained": rate(f_fwd, med_f) / (float(peaks["bf16_tflops_sustained"])
                                                              * ratio)},
        "bwd_main_kernel": None if fp8 else {
            "ms_median": med_b, "ms_mean": statistics.mean(bwd_ms),
            "tflops": rate(f_fwd * BWD_FACTOR, med_b),
            "frac_burst": rate(f_fwd * BWD_FACTOR, med_b) / burst,
            "frac_sustained": rate(f_fwd * BWD_FACTOR, med_b) / float(peaks["bf16_tflops_sustained"]),
            "kernels": "main + deterministic dQ pass" if det else "main"},
        "bwd_pre_and_convert_ms_median": statistics.median(
            sm - fm - bm for sm, fm, bm in zip(kstep_ms, fwd_ms, bwd_ms)),
        "step_ms_median_with_kernel_events": statistics.median(kstep_ms),
    }

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not fp8 and not ext:
        rate, spent, n, threads = oracle_sample_rate(w, t, min_s=10.0, max_s=30.0)
        cpu = {"value": rate, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{n} heads of {w.name}, each cut to its first "
                         f"{min(REF_PREFIX, w.s)} tokens, causal fp64 fwd + bwd, {spent:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "ms_per_step_median": med_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3" if fp8 else "bf16",
            "data": "synthetic (seeded N(0,1) bf16" + (", Q and K x2" if w.qk_mult != 1 else "")
                    + (", encoded as E4M3 with per-tensor descales)" if fp8 else ")"),
            "config": {"workload": w.name, "b": b, "h": h, "s_q": s_q, "s_kv": s, "d": d,
                       "causal": bool(causal), "layout": "bhsd", "variant": variant,
                       **({"h_kv": hk, "mask": ["none", "causal", "causal_bottom_right"][mask],
                           "window_left": window,
                           "flops": "4*d*(visible pairs) fwd, 2.5x bwd"} if ext else {}),
                       "step": ("FP8 fwd (O bf16, LSE, amax)" if fp8 else
                                "fwd (O, LSE) + bwd (dQ, dK, dV)"
                                + (", deterministic dQ pass" if det else "")),
                       "flops_per_step": f_step, "pct_of_peak": 100.0 * value / world / peak,
                       "peak_tflops": peak,
                       "l2": "a 512 MiB buffer (> L2) is written between timed steps; "
                             "inputs+outputs total %d MiB" % ((4 * q.numel() + 2 * k.numel() * 2)
                                                              * 2 >> 20),
                       "parallelism": f"replicas x{world}"},
            "clocks": clocks, "e2e": e2e,
            # both timed loops: K steps for the value, K more with the kernel timer
            "gpu_launches": (1 if fp8 else 4) * 2 * args.steps,
            "roofline": roofline, "phases": phases, "cpu_baseline": cpu,
            "library": version,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_configs(args):
    """Forward and backward chain of every configured workload (dense and
    packed): CUDA events around each call with a 512 MiB L2 flush before it,
    median of 15; the main kernels alone through the kernel timer, median of 11."""
    import torch

    import sdpa_inputs
    import scaled_dot_product_04_gb300 as sdpa
    sdpa.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    names = [args.only] if args.only else list(sdpa_inputs.WORKLOADS)
    for name in names:
        w = sdpa_inputs.WORKLOADS[name]
        t = sdpa_inputs.make(w)
        q, k, v, do = (t[x].to(dev) for x in ("q", "k", "v", "do"))
        if w.layout == "bhsd":
            def fwd():
                return sdpa.attention(q, k, v, scale=w.scale, causal=w.causal)
            o, lse = fwd()

            def bwd():
                return sdpa.attention_bwd(q, k, v, o, do, lse, scale=w.scale, causal=w.causal)
            flops = fwd_flops(w)
        else:
            lens, cu = t["lengths"], t["cu_q"].to(dev)

            def fwd():
                return sdpa.attention_varlen(q, k, v, cu, cu, max(lens), max(lens),
                                             scale=w.scale, causal=w.causal)
            o, lse = fwd()

            def bwd():
                return sdpa.attention_varlen_bwd(q, k, v, o, do, lse, cu, cu, max(lens),
                                                 max(lens), scale=w.scale, causal=w.causal)
            flops = sum(4.0 * w.h * n * n * w.d * (0.5 if w.causal else 1.0) for n in lens)
        if args.probe:
            for _ in range(3):
                fwd()
                bwd()
            torch.cuda.synchronize(dev)
            continue

        def call_ms(fn, iters=15):
            for _ in range(3):
                fn()
            ts = []
            for _ in range(iters):
                flush.zero_()
                a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                fn()
                z.record()
                torch.cuda.synchronize(dev)
                ts.append(a.elapsed_time(z))
            return statistics.median(ts)

        def kernel_ms(fn, iters=11):
            ts = []
            for _ in range(iters):
                flush.zero_()
                a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                sdpa.sdpa_set_kernel_timer(a, z)
                fn()
                sdpa.sdpa_set_kernel_timer(None, None)
                torch.cuda.synchronize(dev)
                ts.append(a.elapsed_time(z))
            return statistics.median(ts)

        f_ms, fk_ms, b_ms, bk_ms = call_ms(fwd), kernel_ms(fwd), call_ms(bwd), kernel_ms(bwd)
        sdpa.sdpa_check_device_error()
        print(json.dumps({
            "workload": name, "fwd_flops": flops, "bwd_flops": BWD_FACTOR * flops,
            "fwd_ms": f_ms, "fwd_kernel_ms": fk_ms, "fwd_tflops": flops / f_ms / 1e9,
            "bwd_chain_ms": b_ms, "bwd_main_ms": bk_ms,
            "bwd_chain_tflops": BWD_FACTOR * flops / b_ms / 1e9,
            "bwd_main_tflops": BWD_FACTOR * flops / bk_ms / 1e9,
            "library": sdpa.sdpa_version()}), flush=True)


def main():
    args = parse_args()
    if args.configs:
        return run_configs(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
