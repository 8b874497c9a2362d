#!/usr/bin/env python
"""Attention fwd+bwd TFLOP/s on one GB300 (and N GPUs as independent replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one pass of the whole path over one batch: fa_fwd (O, logsumexp)
then fa_bwd (dQ, dK, dV) on the headline workload B=2, H=16, N=8192, d=128,
non-causal, bf16 inputs drawn i.i.d. N(0,1) from a fixed seed.  FLOPs per
step: 4*B*H*N^2*d forward + 2.5x that backward.  Rank 0 prints one JSON line.

--impl reference times the fp64 CPU oracle on the host cores instead: each
step is fwd+bwd of a bounded sample of query rows of one head (all keys),
sized so the whole run stays within a few minutes.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd+bwd TFLOP/s at 1 GB300 and fraction of BF16 tensor peak"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--causal", action="store_true", help="time the causal variant of the workload")
    ap.add_argument("--N", type=int, default=8192)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--workload", choices=["sweep", "fwd_b8h16n2048d64", "causal_b4h32n4096d128",
                                           "long_b1h16n16384d128x2", "bnhd_b2h16n8192d128",
                                           "varlen_t16384h16d128_causal", "decode_b16h16nk16384d128",
                                           "decode_b16h16nq8nk16384d128", "fp8_b2h16n8192d128"],
                    default="sweep",
                    help="a named workload instead of the sweep point given by --N/--d/--causal "
                         "(the forward-only one times the forward alone)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="time fwd and bwd separately over the sequence-length sweep (one JSON line per point)")
    return ap.parse_args()


def workload(args):
    from exact_attention_48_gb300 import inputs
    named = {"fwd_b8h16n2048d64": inputs.FWD_B8H16N2048D64, "causal_b4h32n4096d128": inputs.CAUSAL_B4H32N4096D128,
             "long_b1h16n16384d128x2": inputs.LONG_B1H16N16384D128,
             "bnhd_b2h16n8192d128": inputs.BNHD_B2H16N8192D128,
             "varlen_t16384h16d128_causal": inputs.VARLEN_T16384H16D128,
             "decode_b16h16nk16384d128": inputs.DECODE_B16H16NK16384D128,
             "decode_b16h16nq8nk16384d128": inputs.DECODE_B16H16NQ8NK16384D128,
             "fp8_b2h16n8192d128": inputs.FP8_B2H16N8192D128}
    if getattr(args, "workload", "sweep") != "sweep":
        return named[args.workload]
    return inputs.sweep(args.N, args.d, args.causal)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return {k: float(j[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms (a timed
    region of a few tens of steps lasts about a tenth of a second)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.idx)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if ts < t0 or ts > t1 + 0.25:
                continue
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle

def oracle_sample(w, rows, seed_offset=0, nthreads=None):
    """Time the oracle on `rows` query rows of head (0, 0) against all keys.

    Returns (seconds, flops, threads).  FLOPs are counted like the GPU's:
    4*rows*N*d forward and 2.5x that backward (non-causal sample)."""
    import torch
    import oracle
    from exact_attention_48_gb300.inputs import draw_shape
    q, k, v, do = draw_shape(1, 1, w.N, w.d, w.seed + seed_offset, w.input_mult, "cpu", torch.bfloat16)
    q, do = q[:, :, :rows], do[:, :, :rows]
    nt = nthreads or oracle.default_threads()
    qn, kn, vn, don = (oracle._f64(x) for x in (q, k, v, do))
    t0 = time.perf_counter()
    oracle.fwd(qn, kn, vn, False, w.scale, nthreads=nt)
    oracle.bwd(qn, kn, vn, don, False, w.scale, nthreads=nt)
    dt = time.perf_counter() - t0
    flops = 4.0 * rows * w.N * w.d * 3.5
    return dt, flops, nt


def oracle_decode_sample(w, heads, target_s, nthreads=None):
    """Time the oracle's forward over `heads` heads of the decode workload
    (nq query rows against all N cached keys each), repeated until about
    target_s seconds have passed.  Returns (seconds, flops, threads, calls)."""
    import torch
    import oracle
    nt = nthreads or oracle.default_threads()
    g = torch.Generator()
    g.manual_seed(int(w.seed) + 77)
    k, v = (torch.randn((heads, w.N, w.d), generator=g).to(torch.bfloat16) for _ in range(2))
    q = torch.randn((heads, w.nq, w.d), generator=g).to(torch.bfloat16)
    qn, kn, vn = (oracle._f64(x) for x in (q, k, v))
    calls, t0 = 0, time.perf_counter()
    while True:
        oracle.fwd(qn, kn, vn, False, w.scale, nthreads=nt)
        calls += 1
        dt = time.perf_counter() - t0
        if dt >= target_s:
            break
    return dt, calls * 4.0 * heads * w.nq * w.N * w.d, nt, calls


def oracle_fp8_sample(w, rows, nthreads=None):
    """Time the oracle's FP8 forward on `rows` query rows of head (0, 0)
    against all N keys.  Returns (seconds, flops, threads)."""
    import oracle
    from exact_attention_48_gb300.inputs import draw_fp8
    q8, k8, v8, sc = draw_fp8(1, 1, w.N, w.d, w.seed, w.input_mult, "cpu")
    nt = nthreads or oracle.default_threads()
    t0 = time.perf_counter()
    oracle.fwd_fp8(q8[0, 0, :rows], k8[0, 0], v8[0, 0], *sc, False, w.scale, nthreads=nt)
    dt = time.perf_counter() - t0
    return dt, 4.0 * rows * w.N * w.d, nt


def cpu_baseline(w, target_s=12.0):
    if w.layout == "fp8":
        dt, fl, nt = oracle_fp8_sample(w, 64)
        for _ in range(2):  # (two passes, as below)
            rows = int(min(w.N, max(64, target_s * fl / max(dt, 1e-6) / (4.0 * w.N * w.d))))
            dt, fl, nt = oracle_fp8_sample(w, rows)
            if dt >= 0.5 * target_s or rows >= w.N:
                break
        return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": nt, "kind": "oracle",
                "sample": f"FP8 forward of query rows 0..{rows - 1} of head (0,0) against all {w.N} keys, "
                          f"d={w.d}, fp64 C oracle (e4m3 definition), {dt:.1f} s"}
    if w.layout == "decode":
        heads = min(w.B * w.H, 16)
        dt, fl, nt, calls = oracle_decode_sample(w, heads, target_s)
        return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": nt, "kind": "oracle",
                "sample": f"forward of {heads} of the {w.B * w.H} heads ({w.nq} query row(s) against all {w.N} "
                          f"cached keys, d={w.d}), repeated {calls} times, fp64 C oracle, {dt:.1f} s"}
    # calibrate on a small sample, then size the timed one to ~target_s (a
    # second pass: the small sample's rate understates the threads' rate on
    # a larger one)
    dt, fl, nt = oracle_sample(w, 64)
    rows = 64
    for _ in range(2):
        rate = fl / max(dt, 1e-6)
        rows = int(min(w.N, max(64, target_s * rate / (4.0 * w.N * w.d * 3.5))))
        rows = max(64, rows // 64 * 64)
        dt, fl, nt = oracle_sample(w, rows)
        if dt >= 0.5 * target_s or rows >= w.N:
            break
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": nt, "kind": "oracle",
            "sample": f"fwd+bwd of query rows 0..{rows - 1} of head (0,0) against all {w.N} keys, "
                      f"d={w.d}, non-causal, fp64 C oracle, {dt:.1f} s"}


def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    w = workload(args)
    if w.layout == "decode":
        return run_reference_decode(args, w)
    if w.layout == "fp8":
        return run_reference_fp8(args, w)
    # size each step so that warmup + steps take about 100 s in all
    dt, fl, nt = oracle_sample(w, 64)
    rate = fl / max(dt, 1e-6)
    per_step_s = max(0.5, min(10.0, 100.0 / max(1, args.steps + args.warmup)))
    rows = int(min(w.N, max(16, per_step_s * rate / (4.0 * w.N * w.d * 3.5))))
    for i in range(args.warmup):
        oracle_sample(w, rows, i + 1, nt)
    t_total, fl_total = 0.0, 0.0
    for i in range(args.steps):
        dt, fl, _ = oracle_sample(w, rows, 1000 + i, nt)
        t_total += dt
        fl_total += fl
    value = fl_total / t_total / 1e12
    sample = (f"per step: fwd+bwd of {rows} query rows of one head against all {w.N} keys, d={w.d}, "
              f"non-causal, fp64 C oracle")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(w),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nt, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference_fp8(args, w):
    per_step_s = max(0.5, min(10.0, 100.0 / max(1, args.steps + args.warmup)))
    dt, fl, nt = oracle_fp8_sample(w, 32)
    rows = int(min(w.N, max(8, per_step_s * fl / max(dt, 1e-6) / (4.0 * w.N * w.d))))
    for _ in range(args.warmup):
        oracle_fp8_sample(w, rows, nt)
    t_total, fl_total = 0.0, 0.0
    for _ in range(args.steps):
        dt, fl, _ = oracle_fp8_sample(w, rows, nt)
        t_total += dt
        fl_total += fl
    value = fl_total / t_total / 1e12
    sample = (f"per step: FP8 forward of {rows} query rows of one head against all {w.N} keys, d={w.d}, "
              f"fp64 C oracle (e4m3 definition)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(w),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nt, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference_decode(args, w):
    per_step_s = max(0.5, min(10.0, 100.0 / max(1, args.steps + args.warmup)))
    heads = min(w.B * w.H, 16)
    for _ in range(args.warmup):
        oracle_decode_sample(w, heads, per_step_s)
    t_total, fl_total, nt = 0.0, 0.0, 1
    for _ in range(args.steps):
        dt, fl, nt, _ = oracle_decode_sample(w, heads, per_step_s)
        t_total += dt
        fl_total += fl
    value = fl_total / t_total / 1e12
    sample = (f"per step: forward of {heads} heads ({w.nq} query row(s) against all {w.N} cached keys, d={w.d}), "
              f"repeated for about {per_step_s:.1f} s, fp64 C oracle")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(w),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nt, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ multi-rank

def reduce_max(x: float, device=None) -> float:
    """Max of a per-rank float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(flops_per_step_per_rank: float, steps: int, local_ms: float, world: int,
                         device=None) -> tuple[float, float]:
    """Whole-job TFLOP/s (every rank runs its own batch) and the max-over-ranks time in ms."""
    ms = reduce_max(local_ms, device)
    return world * flops_per_step_per_rank * steps / (ms * 1e-3) / 1e12, ms


# ------------------------------------------------------------------ GPU

def token_rows(w):
    """Rows of one head over the whole batch (B*N, or the packed total)."""
    return sum(w.lengths) if w.layout == "varlen" else w.B * w.N


def touched_bytes(w):
    if w.layout == "decode":  # the cache (k, v) plus q, o and lse
        return 2 * w.B * w.H * w.N * w.d * 2 + w.B * w.H * w.nq * (2 * w.d * 2 + 4)
    if w.layout == "fp8":  # q, k, v one byte per element, o bf16, lse
        return w.B * w.H * w.N * (3 * w.d + 2 * w.d + 4)
    n_t = 8 if w.backward else 4  # q, k, v, o (+ dO, dQ, dK, dV)
    return n_t * token_rows(w) * w.H * w.d * 2 + token_rows(w) * w.H * 4


def needs_flush(w):
    return touched_bytes(w) < 2 * L2_BYTES


def config_of(w):
    touched = touched_bytes(w)
    l2 = (f"no flush: the tensors touched per step ({touched / 2**20:.0f} MiB) are larger than the 129 MB L2"
          if not needs_flush(w) else
          f"L2 flushed between steps (a 256 MiB write); the tensors touched per step ({touched / 2**20:.0f} MiB) "
          f"would fit in L2; value = work / sum of the per-step CUDA-event times")
    shape = f"B{w.B} H{w.H} N{w.N} d{w.d}"
    if w.layout == "bnhd":
        shape += " stored [B, N, H, d]"
    elif w.layout == "varlen":
        shape = f"T{token_rows(w)} ({w.B} packed sequences, longest {w.N}) H{w.H} d{w.d}"
    elif w.layout == "decode":
        shape = f"B{w.B} H{w.H} Nq{w.nq} against a cache of Nk{w.N} d{w.d}"
    elif w.layout == "fp8":
        shape = f"B{w.B} H{w.H} N{w.N} d{w.d} e4m3 inputs"
    c = {"workload": f"{'fwd+bwd' if w.backward else 'fwd'} {shape} "
                     f"{'causal' if w.causal else 'non-causal'}{'' if w.layout == 'fp8' else ' bf16'}",
         "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal, "scale": w.scale,
         "layout": w.layout,
         "inputs": (f"i.i.d. N(0,1) x{w.input_mult:g}, per-tensor e4m3 (scale amax/448), seed {w.seed}"
                    if w.layout == "fp8" else f"i.i.d. N(0,1) x{w.input_mult:g} bf16, seed {w.seed}"),
         "l2": l2}
    if w.layout == "varlen":
        c["lengths"] = list(w.lengths)
    if w.layout == "decode":
        c["Nq"] = w.nq
    return c


class Problem:
    """Device tensors of one workload in its storage layout, and the calls
    of the public API that run the path on them.

    ``inputs`` (q, k, v, dO) and ``outputs`` (o, dq, dk, dv) are the storage
    tensors (what a caller copies); ``fwd``/``bwd`` take storage tensors and
    hand the API the views it expects."""

    def __init__(self, w, device="cuda"):
        import torch
        import exact_attention_48_gb300 as fa
        from exact_attention_48_gb300.inputs import draw, draw_shape
        self.w = w
        if w.layout == "decode":
            g = torch.Generator(device=device)
            g.manual_seed(int(w.seed))
            k, v = (torch.randn((w.B, w.H, w.N, w.d), generator=g, device=device).to(torch.bfloat16)
                    for _ in range(2))
            q = torch.randn((w.B, w.H, w.nq, w.d), generator=g, device=device).to(torch.bfloat16)
            self.inputs = [q, k, v, None]
            self.outputs = [torch.empty_like(q), None, None, None]
            self.lse_shape = (w.B, w.H, w.nq)
            self.lse = torch.empty(self.lse_shape, device=device, dtype=torch.float32)
            self.ws = torch.empty(max(1, fa.fa_decode_workspace_bytes(w.B, w.H, w.nq, w.N, w.d)), device=device,
                                  dtype=torch.uint8)
            self._fa = fa
            return
        if w.layout == "fp8":
            from exact_attention_48_gb300.inputs import draw_fp8
            q8, k8, v8, self.fp8_scales = draw_fp8(w.B, w.H, w.N, w.d, w.seed, w.input_mult, device)
            self.inputs = [q8, k8, v8, None]
            self.outputs = [torch.empty(q8.shape, device=device, dtype=torch.bfloat16), None, None, None]
            self.lse_shape = (w.B, w.H, w.N)
            self.lse = torch.empty(self.lse_shape, device=device, dtype=torch.float32)
            self.ws = None
            self._fa = fa
            return
        if w.layout == "varlen":
            T = token_rows(w)
            q, k, v, do = draw_shape(1, w.H, T, w.d, w.seed, w.input_mult, device)
            self.inputs = [x[0].transpose(0, 1).contiguous() for x in (q, k, v, do)]  # [T, H, d]
            offs = [0]
            for n in w.lengths:
                offs.append(offs[-1] + n)
            self.cu = torch.tensor(offs, dtype=torch.int32, device=device)
            self.lse_shape = (w.H, T)
        else:
            q, k, v, do = draw(w, device=device)
            if w.layout == "bnhd":
                self.inputs = [x.transpose(1, 2).contiguous() for x in (q, k, v, do)]  # [B, N, H, d]
            else:
                self.inputs = [q, k, v, do]
            self.lse_shape = (w.B, w.H, w.N)
        self.outputs = [torch.empty_like(self.inputs[0]) for _ in range(4)]
        self.lse = torch.empty(self.lse_shape, device=device, dtype=torch.float32)
        self.ws = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.N, w.d), device=device, dtype=torch.uint8)
        self._fa = fa

    def view(self, x):
        return x.transpose(1, 2) if self.w.layout == "bnhd" else x

    def fwd(self, q, k, v, o, lse):
        w, fa, V = self.w, self._fa, self.view
        if w.layout == "decode":
            fa.fa_fwd_decode(q, k, v, None, w.causal, w.scale, o=o, lse=lse, workspace=self.ws)
        elif w.layout == "fp8":
            fa.fa_fwd_fp8(q, k, v, *self.fp8_scales, w.causal, w.scale, o=o, lse=lse)
        elif w.layout == "varlen":
            fa.fa_fwd_varlen(q, k, v, self.cu, w.N, w.causal, w.scale, o=o, lse=lse)
        elif w.layout == "bnhd":
            fa.fa_fwd_strided(V(q), V(k), V(v), w.causal, w.scale, o=V(o), lse=lse)
        else:
            fa.fa_fwd(q, k, v, w.causal, w.scale, o=o, lse=lse)

    def bwd(self, q, k, v, o, do, lse, dq, dk, dv):
        w, fa, V = self.w, self._fa, self.view
        if w.layout == "varlen":
            fa.fa_bwd_varlen(q, k, v, o, do, lse, self.cu, w.N, w.causal, w.scale, dq=dq, dk=dk, dv=dv,
                             workspace=self.ws)
        elif w.layout == "bnhd":
            fa.fa_bwd_strided(V(q), V(k), V(v), V(o), V(do), lse, w.causal, w.scale, dq=V(dq), dk=V(dk),
                              dv=V(dv), workspace=self.ws)
        else:
            fa.fa_bwd(q, k, v, o, do, lse, w.causal, w.scale, dq=dq, dk=dk, dv=dv, workspace=self.ws)


def traffic_record(kernel: str, workload_name: str):
    """DRAM bytes per launch from the committed ncu summary, or None if the
    kernel source changed since those counters were taken or they were taken
    on another workload."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f).get(kernel)
    except Exception:
        return None
    if not rec:
        return None
    src = os.path.join(ROOT, rec["source"])
    try:
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    if h != rec.get("source_sha256_16"):
        return None
    if rec.get("workload") != workload_name:
        return None
    return float(rec["bytes_per_launch"])


def run_ours(args):
    import torch

    world, rank, local = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (there is no CPU fallback)")
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from exact_attention_48_gb300 import fa_device_status
    from exact_attention_48_gb300.binding import fa_debug_time_next_bwd

    w = workload(args)
    # every rank runs its own batch (independent heads): weak scaling, no data-path collective
    pb = Problem(w)
    q, k, v, do = pb.inputs
    o, dq, dk, dv = pb.outputs
    lse = pb.lse
    stream = torch.cuda.current_stream()

    bwd_on = w.backward  # the forward-only workload times the forward alone

    def step(evs=None, kernel_times=False):
        if evs is not None:
            evs[0].record(stream)
        pb.fwd(q, k, v, o, lse)
        if evs is not None:
            evs[1].record(stream)
        if bwd_on:
            if kernel_times:
                # events between the backward's kernels; the library then runs
                # them one after the other instead of side by side
                fa_debug_time_next_bwd(evs[2], evs[3], evs[4])
            pb.bwd(q, k, v, o, do, lse, dq, dk, dv)
        if evs is not None:
            evs[5].record(stream)

    for _ in range(max(args.warmup, 3 if args.warmup >= 3 else args.warmup)):
        step()
    torch.cuda.synchronize()
    if fa_device_status() != 0:
        raise SystemExit("device status error after warm-up")

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.6)  # let the sampler start
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    flush = torch.empty(256 * 2**20, device="cuda", dtype=torch.uint8) if needs_flush(w) else None
    start.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
        step(evs[i])
    stop.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier()
    clk = clocks.stop(t_wall0, t_wall1)
    if fa_device_status() != 0:
        raise SystemExit("device status error in the timed region")
    # Per-kernel durations for the roofline: a second timed pass with events
    # between the backward's kernels (which makes them run one after the
    # other; the main timed region above runs the dQ kernel next to the
    # dK/dV kernel).
    kevs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(min(args.steps, 50))]
    if bwd_on:
        for i in range(len(kevs)):
            if flush is not None:
                flush.fill_(i & 0xFF)
            step(kevs[i], kernel_times=True)
        torch.cuda.synchronize()

    flops_step = w.flops_fwd() + (w.flops_bwd() if bwd_on else 0.0)
    total_ms = start.elapsed_time(stop)
    if flush is not None:  # leave the flushes out: the steps' own event times
        total_ms = sum(e[0].elapsed_time(e[5]) for e in evs)
    value, elapsed_ms = aggregate_throughput(flops_step, args.steps, total_ms, world, "cuda")
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    if bwd_on:
        bwd_ms = statistics.mean(e[1].elapsed_time(e[5]) for e in evs)
        dkdv_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in kevs)
        dq_ms = statistics.mean(e[3].elapsed_time(e[4]) for e in kevs)

    peaks, peak_src = load_peaks()
    peak_sus, peak_burst = peaks["bf16_tflops_sustained"], peaks["bf16_tflops"]
    peak_note = "bf16"
    if w.layout == "fp8":
        # the 8-bit tensor path: the measured bf16 peaks times the nominal
        # dense ratio of the two formats (4.5 / 2.25 PFLOP/s)
        peak_sus, peak_burst, peak_note = 2.0 * peak_sus, 2.0 * peak_burst, "fp8 = 2 x bf16"
    fwd_tf = w.flops_fwd() / (fwd_ms * 1e-3) / 1e12
    bwd_tf = w.flops_bwd() / (bwd_ms * 1e-3) / 1e12 if bwd_on else None
    # Per-kernel tensor work actually executed (the dense products of each
    # kernel, in units of the forward's 4*B*H*N^2*d): forward 1.0, dK/dV 2.0
    # (S^T, dP^T, dV, dK), dQ 1.5 (S, dP, dQ).  The backward headline keeps
    # the 2.5x count of the metric and credits no recomputation.
    kernels = [("fa_fwd_fp8_kernel" if w.layout == "fp8" else "fa_fwd_kernel", fwd_ms, 1.0 * w.flops_fwd())]
    if bwd_on:
        kernels += [("fa_bwd_dkdv_kernel", dkdv_ms, 2.0 * w.flops_fwd()),
                    ("fa_bwd_dq_kernel", dq_ms, 1.5 * w.flops_fwd())]
    dom, dom_ms, dom_flops = max(kernels, key=lambda k: k[1])
    dom_tf = dom_flops / (dom_ms * 1e-3) / 1e12
    traffic = traffic_record(dom, config_of(w)["workload"])
    # Which measured peak applies: the burst figure (cuBLAS at full clock)
    # unless the SM clock sampled during the timed region sat well below its
    # maximum (the power-capped regime the sustained figure was taken in).
    full_clock = (clk.get("sm_mhz") is None or clk.get("sm_max_mhz") is None
                  or clk["sm_mhz"] >= 0.95 * clk["sm_max_mhz"])
    peak, peak_kind = (peak_burst, "bf16_tflops (burst)") if full_clock else \
        (peak_sus, "bf16_tflops_sustained (SM clock below 95 % of its maximum in the timed region)")

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {"fp8": "e4m3", "decode": "fp32"}.get(w.layout, "bf16"), "data": "synthetic",
        "config": config_of(w),
        "fwd": {"ms": fwd_ms, "tflops": fwd_tf, "frac": fwd_tf / peak, "frac_of_sustained": fwd_tf / peak_sus,
                "frac_of_burst": fwd_tf / peak_burst},
        # the backward's method fraction: 2.5 x the forward's FLOPs (no
        # credit for recomputation) over the time of all its kernels
        "bwd": ({"ms": bwd_ms, "tflops": bwd_tf, "frac_method": bwd_tf / peak,
                 "frac_of_sustained": bwd_tf / peak_sus, "frac_of_burst": bwd_tf / peak_burst} if bwd_on else None),
        "kernels": {name: {"ms": ms, "tensor_tflops_executed": fl / (ms * 1e-3) / 1e12,
                           "frac": fl / (ms * 1e-3) / 1e12 / peak,
                           "frac_of_sustained": fl / (ms * 1e-3) / 1e12 / peak_sus} for name, ms, fl in kernels},
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": dom_tf,
                     "peak": peak, "unit": "TFLOP/s", "frac": dom_tf / peak,
                     "frac_of_burst": dom_tf / peak_burst, "frac_of_sustained": dom_tf / peak_sus,
                     "peak_source": (f"{peak_src} {peak_kind}"
                                     + (", x2 for the fp8 path (nominal fp8/bf16 ratio)" if w.layout == "fp8" else "")),
                     "flops_per_launch": dom_flops, "traffic": traffic},
        "kernel_timing": ("per-kernel durations from a second timed pass of the same steps with events between "
                          "the backward's kernels (which then run one after the other; in the main timed region "
                          "the dQ kernel runs next to the dK/dV kernel on a side stream)") if bwd_on else None,
        "gpu_launches": (4 if bwd_on else 1) * args.steps,  # fwd; bwd pre, dK/dV, dQ
        "clocks": clk,
    }
    if w.layout == "decode":
        # HBM-bound: the roofline is bytes moved (the cache once, q, o, lse)
        # over the call's time (the split kernel and, when the keys are cut
        # into several chunks, the small merge kernel), against the measured
        # copy bandwidth.
        from exact_attention_48_gb300 import fa_decode_workspace_bytes
        nbytes = touched_bytes(w)
        gbs = nbytes / (fwd_ms * 1e-3) / 1e9
        merged = fa_decode_workspace_bytes(w.B, w.H, w.nq, w.N, w.d) > 0
        # (2..8 query rows at d = 128: the tensor-core split kernel)
        kname = "fa_decode_tc_kernel" if (w.d == 128 and w.nq >= 2) else "fa_decode_kernel"
        line["fwd"] = {"ms": fwd_ms, "tflops": fwd_tf, "gbs": gbs}
        line["kernels"] = {kname + (" + fa_decode_combine_kernel" if merged else ""): {"ms": fwd_ms, "gbs": gbs}}
        line["roofline"] = {"bound": "hbm", "kernel": kname, "achieved": gbs, "peak": peaks["hbm_gbs"],
                            "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                            "peak_source": f"{peak_src} hbm_gbs (copy bandwidth)",
                            "bytes_per_launch": nbytes, "timed": "the whole call (split kernel + merge kernel)",
                            "traffic": traffic_record(kname, config_of(w)["workload"])}
        line["gpu_launches"] = (2 if merged else 1) * args.steps

    if not args.no_e2e:
        line["e2e"] = e2e_leg(pb, args, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def e2e_leg(pb, args, world):
    """Same metric through the public API from HOST buffers: every step copies
    q, k, v, dO from pinned host memory to the device and o, lse, dq, dk, dv
    back, inside the timed region.

    Three ways, all reported; the value is the best.  Sequential: copy in,
    compute, copy out, one step after the other on one stream.  Pipelined:
    NSETS sets of device buffers used in turn; step i's inputs are copied in
    on one stream while earlier steps compute, and its outputs copied out on
    a third stream while later steps compute, each copy ordered against the
    compute by events.  Pipelined on one copy stream: the same, with both
    directions' copies in turn on a single stream (the host link's two
    directions then never run at once, which some boxes' host-copy paths
    prefer).  Every step still moves all of its bytes both ways."""
    import torch
    w = pb.w
    q = pb.inputs[0]
    n_in, n_out = (4, 4) if w.backward else (3, 1)
    hin = [t.cpu().pin_memory() for t in pb.inputs[:n_in]]
    steps = max(4, min(args.steps, 20))
    flops = w.flops_fwd() + (w.flops_bwd() if w.backward else 0.0)

    def make_set():
        ins = [torch.empty_like(t) for t in pb.inputs[:n_in]]
        outs = [torch.empty_like(pb.outputs[0])] + [torch.empty_like(q) for _ in range(n_out - 1)]
        lse = torch.empty(pb.lse_shape, device="cuda", dtype=torch.float32)
        hout = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]
        hlse = torch.empty(pb.lse_shape, dtype=torch.float32).pin_memory()
        return ins, outs, lse, hout, hlse

    def compute(ins, outs, lse):
        qq, kk, vv = ins[0], ins[1], ins[2]
        pb.fwd(qq, kk, vv, outs[0], lse)
        if w.backward:
            pb.bwd(qq, kk, vv, outs[0], ins[3], lse, outs[1], outs[2], outs[3])

    # three sets: a copy that starts late (the copy engines and the host
    # share the box with other work) still has a step of slack
    NSETS = 3
    sets = [make_set() for _ in range(NSETS)]
    sc = torch.cuda.current_stream()
    sh, sd = torch.cuda.Stream(), torch.cuda.Stream()

    # sequential
    def seq_step():
        ins, outs, lse, hout, hlse = sets[0]
        for dst, src in zip(ins, hin):
            dst.copy_(src, non_blocking=True)
        compute(ins, outs, lse)
        for dst, src in zip(hout, outs):
            dst.copy_(src, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)

    for _ in range(2):
        seq_step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(sc)
    for _ in range(steps):
        seq_step()
    b.record(sc)
    torch.cuda.synchronize()
    seq_value, _ = aggregate_throughput(flops, steps, a.elapsed_time(b), world, "cuda")

    # pipelined
    h2d_done = [torch.cuda.Event() for _ in range(NSETS)]
    comp_done = [torch.cuda.Event() for _ in range(NSETS)]
    d2h_done = [torch.cuda.Event() for _ in range(NSETS)]

    def pipe_steps(n):
        for i in range(n):
            bset = i % NSETS
            ins, outs, lse, hout, hlse = sets[bset]
            with torch.cuda.stream(sh):
                if i >= NSETS:
                    sh.wait_event(comp_done[bset])  # inputs of step i-NSETS consumed
                for dst, src in zip(ins, hin):
                    dst.copy_(src, non_blocking=True)
                h2d_done[bset].record(sh)
            sc.wait_event(h2d_done[bset])
            if i >= NSETS:
                sc.wait_event(d2h_done[bset])  # outputs of step i-NSETS copied out
            compute(ins, outs, lse)
            comp_done[bset].record(sc)
            with torch.cuda.stream(sd):
                sd.wait_event(comp_done[bset])
                for dst, src in zip(hout, outs):
                    dst.copy_(src, non_blocking=True)
                hlse.copy_(lse, non_blocking=True)
                d2h_done[bset].record(sd)
        sc.wait_stream(sh)
        sc.wait_stream(sd)

    pipe_steps(NSETS)
    torch.cuda.synchronize()
    a2, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a2.record(sc)
    sh.wait_stream(sc)
    sd.wait_stream(sc)
    pipe_steps(steps)
    b2.record(sc)
    torch.cuda.synchronize()
    pipe_value, _ = aggregate_throughput(flops, steps, a2.elapsed_time(b2), world, "cuda")

    # pipelined on one copy stream: in iteration i the copy stream takes
    # step i's inputs, then step i-1's outputs (after step i-1's compute), so
    # step i+1's inputs queue behind them while step i computes
    def one_stream_steps(n):
        for i in range(n + 1):
            if i < n:
                bset = i % NSETS
                ins = sets[bset][0]
                with torch.cuda.stream(sh):
                    if i >= NSETS:
                        sh.wait_event(comp_done[bset])
                    for dst, src in zip(ins, hin):
                        dst.copy_(src, non_blocking=True)
                    h2d_done[bset].record(sh)
            if i >= 1:
                pset = (i - 1) % NSETS
                _, outs, lse, hout, hlse = sets[pset]
                with torch.cuda.stream(sh):
                    sh.wait_event(comp_done[pset])
                    for dst, src in zip(hout, outs):
                        dst.copy_(src, non_blocking=True)
                    hlse.copy_(lse, non_blocking=True)
                    d2h_done[pset].record(sh)
            if i < n:
                bset = i % NSETS
                ins, outs, lse = sets[bset][0], sets[bset][1], sets[bset][2]
                sc.wait_event(h2d_done[bset])
                if i >= NSETS:
                    sc.wait_event(d2h_done[bset])
                compute(ins, outs, lse)
                comp_done[bset].record(sc)
        sc.wait_stream(sh)

    one_stream_steps(NSETS)
    torch.cuda.synchronize()
    a3, b3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a3.record(sc)
    sh.wait_stream(sc)
    one_stream_steps(steps)
    b3.record(sc)
    torch.cuda.synchronize()
    one_value, _ = aggregate_throughput(flops, steps, a3.elapsed_time(b3), world, "cuda")
    h2d = sum(t.numel() * t.element_size() for t in hin)
    d2h = sum(t.numel() * t.element_size() for t in sets[0][3]) + sets[0][4].numel() * 4
    # the best of the three schedules (a copy-bound workload, whose copies
    # cannot hide behind its compute, may do better on one stream)
    best = max(pipe_value, one_value, seq_value)
    schedule = "pipelined" if best == pipe_value else ("pipelined_one_copy_stream" if best == one_value else "sequential")
    return {"value": best, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "pipelined": schedule != "sequential",
            "schedule": schedule, "pipelined_value": pipe_value, "pipelined_one_copy_stream_value": one_value,
            "sequential_value": seq_value,
            "note": "value: the best of three schedules. pipelined_value: over three buffer sets, each step's "
                    "host->device copy overlaps earlier steps' compute and its device->host copy later steps', "
                    "on their own streams; pipelined_one_copy_stream_value: the same with both directions on one "
                    "copy stream; sequential_value: copy in, compute, copy out on one stream"}


def run_sweep(args):
    """B*N = 16384 tokens, H = 16, N in 512..16384, d in {64, 128}, causal and
    not: forward and backward timed separately with CUDA events (median of
    args.steps after args.warmup), one JSON line per point."""
    import torch
    from exact_attention_48_gb300 import fa_bwd, fa_bwd_workspace_bytes, fa_fwd
    from exact_attention_48_gb300.inputs import SWEEP_N, draw, sweep
    peaks, peak_src = load_peaks()
    steps = max(5, min(args.steps, 50))
    for d in (64, 128):
        for causal in (False, True):
            for N in SWEEP_N:
                w = sweep(N, d, causal)
                q, k, v, do = draw(w, device="cuda")
                o, lse = fa_fwd(q, k, v, causal, w.scale)
                ws = torch.empty(fa_bwd_workspace_bytes(w.B, w.H, w.N, w.d), device="cuda", dtype=torch.uint8)
                dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
                for _ in range(max(3, args.warmup)):
                    fa_fwd(q, k, v, causal, w.scale, o=o, lse=lse)
                    fa_bwd(q, k, v, o, do, lse, causal, w.scale, dq=dq, dk=dk, dv=dv, workspace=ws)
                tf, tb = [], []
                for _ in range(steps):
                    e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                    e[0].record()
                    fa_fwd(q, k, v, causal, w.scale, o=o, lse=lse)
                    e[1].record()
                    fa_bwd(q, k, v, o, do, lse, causal, w.scale, dq=dq, dk=dk, dv=dv, workspace=ws)
                    e[2].record()
                    torch.cuda.synchronize()
                    tf.append(e[0].elapsed_time(e[1]))
                    tb.append(e[1].elapsed_time(e[2]))
                mf, mb = statistics.median(tf), statistics.median(tb)
                ftf = w.flops_fwd() / (mf * 1e-3) / 1e12
                btf = w.flops_bwd() / (mb * 1e-3) / 1e12
                # algorithmic HBM bytes of the forward: q, k, v read, o written, lse written;
                # of the backward: q, k, v, o, dO read, dq, dk, dv written, lse read
                fbytes = 8.0 * w.B * w.H * w.N * w.d + 4.0 * w.B * w.H * w.N
                bbytes = 16.0 * w.B * w.H * w.N * w.d + 4.0 * w.B * w.H * w.N
                # roof of each pass: the tensor peak, or the HBM copy bandwidth
                # times the pass's arithmetic intensity where that is lower
                # (short or causal sequences)
                froof = min(peaks["bf16_tflops"], w.flops_fwd() / fbytes * peaks["hbm_gbs"] / 1e3)
                broof = min(peaks["bf16_tflops"], w.flops_bwd() / bbytes * peaks["hbm_gbs"] / 1e3)
                print(json.dumps({"sweep": w.name, "B": w.B, "H": w.H, "N": N, "d": d, "causal": causal,
                                  "fwd_ms": mf, "fwd_tflops": ftf, "fwd_frac_of_burst": ftf / peaks["bf16_tflops"],
                                  "fwd_frac_of_sustained": ftf / peaks["bf16_tflops_sustained"],
                                  "fwd_roof_tflops": froof, "fwd_frac_of_roof": ftf / froof,
                                  "bwd_ms": mb, "bwd_tflops": btf, "bwd_frac_of_burst": btf / peaks["bf16_tflops"],
                                  "bwd_frac_of_sustained": btf / peaks["bf16_tflops_sustained"],
                                  "bwd_roof_tflops": broof, "bwd_frac_of_roof": btf / broof,
                                  "fwd_hbm_gbs_algorithmic": fbytes / (mf * 1e-3) / 1e9,
                                  "bwd_hbm_gbs_algorithmic": bbytes / (mb * 1e-3) / 1e9, "peak_source": peak_src}),
                      flush=True)
                del q, k, v, do, o, lse, ws, dq, dk, dv
                torch.cuda.empty_cache()


def main():
    args = parse_args()
    if args.sweep:
        run_sweep(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
