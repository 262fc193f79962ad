"""Benchmark: exact disentangled attention forward + backward through the C ABI.

One step = df_attn_fwd + df_attn_bwd over one batch of the L=8192 length-sweep
workload (B=2, H=12, D=64, bf16, att_span 256 -> R=512, buckets 256 / max
relative positions 512, 16,384 tokens, N(0,1) synthetic inputs).  Throughput
is counted with the pages' FLOP formula: BH(4L^2 D + 4LRD) forward plus
BH(10L^2 D + 12LRD) backward.  The forward saves the band bias for the
backward (df_attn_params.band_bias), as a training step would.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

N > 1 runs under torchrun, one rank per GPU, each rank its own batch (weak
scaling, no collective on the data path: the batch shards into independent
sequences).  `--impl reference` times the fp64 CPU oracle on host cores on a
bounded row sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "sweep_L8192"
PHASES = ("fwd", "dq", "dkv", "rel")


def flops_fwd(B, H, L, D, R):
    return B * H * (4 * L * L * D + 4 * L * R * D)


def flops_bwd(B, H, L, D, R):
    return B * H * (10 * L * L * D + 12 * L * R * D)


def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own batch (weak scaling: independent sequences)."""
    return base_seed + rank


def max_over_ranks(x: float, world: int, device) -> float:
    """Slowest rank's value (the job's time is the slowest replica's)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, step_flops: float, seconds_per_step: float) -> float:
    """Whole-job TFLOP/s: every rank processed step_flops per step."""
    return world * step_flops / seconds_per_step / 1e12


# DRAM traffic of one launch of each attention kernel at this workload, from the
# committed ncu summary of that kernel; reported only while the kernel's sources
# are the ones the counters were taken on (else null)
PROFILE_FILES = {
    "fwd": ("fwd_tc_kernel_L8192_B1_H12_D64.md", ["df_fwd.cu", "df_tile.cuh", "df_common.cuh"]),
    "dkv": ("bwd_tc_kernel_dkv_L8192_B1_H12_D64.md",
            ["df_bwd_kernel.cuh", "df_bwd_dkv.cu", "df_tile.cuh", "df_common.cuh"]),
    "dq": ("bwd_tc_kernel_dq_L8192_B1_H12_D64.md",
           ["df_bwd_kernel.cuh", "df_bwd_dq.cu", "df_tile.cuh", "df_common.cuh"]),
}


def kernel_traffic(kernel: str):
    import hashlib
    if kernel == "bwd_attn":   # the concurrent dQ + dK/dV pair: both kernels' traffic
        a, b = kernel_traffic("dq"), kernel_traffic("dkv")
        return None if a is None or b is None else a + b
    if kernel not in PROFILE_FILES:
        return None
    md, srcs = PROFILE_FILES[kernel]
    try:
        fields = {}
        with open(os.path.join(ROOT, "profiles", md)) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip().split()[0] if v.strip() else ""
        h = hashlib.sha256()
        for name in srcs:
            with open(os.path.join(ROOT, "exact_deberta_disentangled_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
        if fields.get("kernel_source_sha256_16") != h.hexdigest()[:16]:
            return None
        return int(fields["traffic_bytes_per_launch_L8192_B2"])
    except Exception:
        return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def oracle_sample(target_s: float, seed_offset: int = 0):
    """Time the fp64 oracle (as it stands) on a row sample of the workload:
    query rows [0, r) of one (sequence, head) pair per host thread.  Returns
    (TFLOP/s by the pages' count, description, threads)."""
    import numpy as np

    from exact_deberta_disentangled_gb300 import synth
    from oracle import oracle

    w = synth.WORKLOADS[WORKLOAD]
    x = synth.make_inputs(w)
    prob = oracle.Problem(x.cu_seqlens.numpy(), w.H, w.D, w.span, w.nb, w.mp)
    f64 = lambda a: a.double().numpy()
    args = [f64(a) for a in (x.q, x.k, x.v, x.qr, x.kr, x.dout)]
    nthr = oracle.max_threads()
    pairs = [(p // w.H % x.B, p % w.H) for p in range(nthr)]
    # calibrate on a few rows, then size the sample to the time target
    t = time.perf_counter()
    oracle.step_rows_sample(prob, pairs, 0, 8, *args, nthreads=nthr)
    per_row = max((time.perf_counter() - t) / 8, 1e-4)
    rows = int(max(8, min(w.L, target_s / per_row)))
    t = time.perf_counter()
    oracle.step_rows_sample(prob, pairs, 0, rows, *args, nthreads=nthr)
    dt = time.perf_counter() - t
    L, D, R = w.L, w.D, w.R
    per_row_flops = (4 * L * D + 4 * R * D) + (10 * L * D + 12 * R * D)
    flops = per_row_flops * rows * len(pairs)
    desc = (f"fp64 oracle fwd+bwd of query rows 0..{rows - 1} of {len(pairs)} (sequence, head) pairs of the "
            f"L={L} workload, one pair per thread; pages' FLOP count per row")
    return flops / dt / 1e12, desc, nthr, dt


def run_reference(args, rank, world):
    if rank != 0:
        return
    vals = []
    desc, nthr = "", 0
    for i in range(args.warmup + args.steps):
        v, desc, nthr, _ = oracle_sample(args.ref_seconds)
        if i >= args.warmup:
            vals.append(v)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "length sweep L=8192: B=2, H=12, D=64, att_span=256 (R=512), buckets 256, "
                               "max_rel 512, 16384 tokens", "sample": desc},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nthr, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


METRIC = "disentangled attn fwd+bwd TFLOP/s (pages' FLOP count) at L=8192 bf16, % roofline"


def run_gpu(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from exact_deberta_disentangled_gb300 import binding as Bd
    from exact_deberta_disentangled_gb300 import build as build_mod
    from exact_deberta_disentangled_gb300 import synth

    if not os.path.exists(Bd.LIB_PATH):
        if rank == 0:
            build_mod.build()
        if world > 1:
            dist.barrier()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[WORKLOAD]
    x = synth.make_inputs(w, seed=rank_seed(w.seed, rank))
    B, L, H, D, R = x.B, x.L, w.H, w.D, w.R
    g = Bd.Geometry(B=B, L=L, H=H, D=D, span=w.span, nb=w.nb, mp=w.mp)
    q, k, v, qr, kr, do = [t.to(dev) for t in (x.q, x.k, x.v, x.qr, x.kr, x.dout)]
    g.band_bias = Bd.alloc_band_bias(g, q.dtype, dev)   # saved by the forward, read by the backward
    out = torch.empty_like(q)
    lse = torch.empty(g.lse_shape(), dtype=torch.float32, device=dev)
    grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(qr),
             torch.empty_like(kr))
    wsf = Bd.alloc_workspace(g, q.dtype, False, dev)
    wsb = Bd.alloc_workspace(g, q.dtype, True, dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)   # > 2x L2
    stream = torch.cuda.current_stream()

    def step():
        Bd.attn_fwd(g, q, k, v, qr, kr, out=out, lse=lse, workspace=wsf)
        Bd.attn_bwd(g, q, k, v, qr, kr, out, lse, do, grads=grads, workspace=wsb)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert Bd.device_error(wsf) == 0 and Bd.device_error(wsb) == 0

    # per-kernel timing hooks (CUDA events recorded by the library on this stream)
    ev_ph = [torch.cuda.Event(enable_timing=True) for _ in range(2 * len(PHASES))]
    for e in ev_ph:
        e.record(stream)
    torch.cuda.synchronize()
    phase_ms = {p: [] for p in PHASES}
    phase_ms["bwd_attn"] = []   # dQ and dK/dV run concurrently: first start to last end
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    Bd.set_profile_events(ev_ph)
    try:
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
            torch.cuda.synchronize()
            for pi, p in enumerate(PHASES):
                phase_ms[p].append(ev_ph[2 * pi].elapsed_time(ev_ph[2 * pi + 1]))
            # the dQ kernel (side stream) and the dK/dV kernel (this stream) overlap
            s_dq, e_dq, s_dkv, e_dkv = ev_ph[2], ev_ph[3], ev_ph[4], ev_ph[5]
            t_dkv0, t_dq1, t_dkv1 = (s_dq.elapsed_time(x) for x in (s_dkv, e_dq, e_dkv))
            phase_ms["bwd_attn"].append(max(t_dq1, t_dkv1) - min(0.0, t_dkv0))
    finally:
        Bd.set_profile_events(None)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    # a bounded wait that gave up inside a kernel leaves its code in the
    # workspace's error word: such a step did not do its work
    ef, eb = Bd.device_error(wsf), Bd.device_error(wsb)
    if ef or eb:
        raise SystemExit(f"device error word after the timed steps: forward {ef}, backward {eb}")
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    step_q = quantiles(step_ms)
    print("per-step ms: " + " ".join(f"{t:.3f}" for t in step_ms) + " | fwd: " +
          " ".join(f"{t:.3f}" for t in phase_ms["fwd"]), file=sys.stderr, flush=True)
    ms = sum(step_ms) / len(step_ms)
    ms = max_over_ranks(ms, world, dev)
    fl_f, fl_b = flops_fwd(B, H, L, D, R), flops_bwd(B, H, L, D, R)
    step_flops = fl_f + fl_b
    value = job_throughput(world, step_flops, ms * 1e-3)

    # end-to-end through df_attn_step_host: pinned host buffers, copies inside the timed region
    hq, hk, hv, hqr, hkr, hdo = [t.pin_memory() for t in (x.q, x.k, x.v, x.qr, x.kr, x.dout)]
    houts = (torch.empty_like(hq).pin_memory(), torch.empty(g.lse_shape(), dtype=torch.float32).pin_memory(),
             torch.empty_like(hq).pin_memory(), torch.empty_like(hk).pin_memory(),
             torch.empty_like(hv).pin_memory(), torch.empty_like(hqr).pin_memory(),
             torch.empty_like(hkr).pin_memory())
    arena = torch.empty(Bd.step_host_arena_size(g, q.dtype), dtype=torch.uint8, device=dev)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hqr, hkr, hdo))
    d2h = sum(t.numel() * t.element_size() for t in houts)
    for _ in range(max(1, args.warmup // 2)):
        Bd.step_host(g, hq, hk, hv, hqr, hkr, hdo, houts, arena)
    e2e_steps = max(3, args.steps // 2)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        Bd.step_host(g, hq, hk, hv, hqr, hkr, hdo, houts, arena)
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    e2e_s = max_over_ranks(e2e_s, world, dev)
    e2e_value = job_throughput(world, step_flops, e2e_s)

    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    avg = {p: sum(v) / len(v) for p, v in phase_ms.items()}
    # roofline units: the forward kernel, the concurrent dQ + dK/dV pair, the
    # relative-gradient kernels
    dominant = max(("fwd", "bwd_attn", "rel"), key=lambda p: avg[p])
    # algorithmic tensor FLOPs of each kernel by the pages' count:
    #   fwd kernel  4 L^2 D + 4 L R D (all of the forward count)
    #   dK/dV kernel  S^T, dP^T, dV, dK products: 8 L^2 D
    #   dQ kernel     dQ product: 2 L^2 D (its recomputed S, dP are not credited)
    #   rel           the relative-position gradient half on the caller's
    #                 stream after the dK/dV kernel (dK += G' Qr, dQr): 4 L R D
    #   bwd_attn      the dQ and dK/dV kernels, which run concurrently, and the
    #                 other relative half (dQ += G Kr, dKr), which runs on the
    #                 dQ kernel's stream inside the same window: 10 L^2 D + 4 L R D
    kflops = {"fwd": fl_f, "dkv": B * H * 8 * L * L * D, "dq": B * H * 2 * L * L * D,
              "rel": B * H * 4 * L * R * D, "bwd_attn": B * H * (10 * L * L * D + 4 * L * R * D)}
    peak = peaks.get("bf16_tflops", 1900.0)
    achieved = kflops[dominant] / (avg[dominant] * 1e-3) / 1e12
    traffic = kernel_traffic(dominant)
    extras = None
    if not args.no_extras:
        extras = run_extras(dev, args.extra_iters, 3, flush)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        v_cpu, desc, nthr, _ = oracle_sample(args.ref_seconds)
        cpu = {"value": v_cpu, "unit": "TFLOP/s", "cores": nthr, "kind": "oracle", "sample": desc}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "step_ms_quantiles": step_q, "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "length sweep L=8192: B=2, H=12, D=64, att_span=256 (R=512), buckets 256, "
                               "max_rel 512, 16384 tokens per GPU, N(0,1) inputs", "global_batch": B * world,
                   "seq_len": L, "parallelism": f"replicas x{world} (independent batches)",
                   "l2": "flushed before every timed step (512 MB write)",
                   "flops_per_step": step_flops, "fwd_flops": fl_f, "bwd_flops": fl_b,
                   "pct_of_bf16_peak": 100.0 * (value / world) / peak},
        "roofline": {"bound": "tensor", "kernel": dominant, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_src} bf16_tflops (burst)",
                     "kernel_ms": avg, "kernel_flops": kflops},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_s * 1e3},
        # per step: delta table x2, relative scalars x2, fwd, Dl, dQ, dK/dV,
        # relative-gradient row / column / reduce kernels x2 each
        "gpu_launches": args.steps * 14,
        "clocks": clk,
        "extras": extras,
    }
    print(json.dumps(line), flush=True)


def quantiles(ts):
    """min / p10 / median / p90 of a list of per-iteration times (ms)."""
    import numpy as np
    a = np.asarray(ts, dtype=np.float64)
    return {"min": float(a.min()), "p10": float(np.percentile(a, 10)), "median": float(np.median(a)),
            "p90": float(np.percentile(a, 90)), "n": int(a.size)}


def workload_flops(x, w, H):
    """The pages' FLOP count of one call: per (sequence, head) of length l,
    4 l^2 D + 4 l R D forward and 10 l^2 D + 12 l R D backward; padded
    workloads are counted on the padded length (every tile is computed)."""
    lens = (x.cu_seqlens[1:] - x.cu_seqlens[:-1]).tolist()
    D, R = w.D, w.R
    f = sum(H * (4 * l * l * D + 4 * l * R * D) for l in lens)
    b = sum(H * (10 * l * l * D + 12 * l * R * D) for l in lens)
    return f, b


def time_phases(name, dev, iters, warmup, flush, fp32_fast=False, **make_kw):
    """Forward, backward (alone, from the saved forward outputs) and forward +
    backward of one workload through the C ABI: per-iteration CUDA-event
    times on the launching stream, L2 flushed before every iteration
    (fp32_fast: fp32 tensors in the fast mode)."""
    import torch

    from exact_deberta_disentangled_gb300 import binding as Bd
    from exact_deberta_disentangled_gb300 import synth

    w = synth.WORKLOADS[name]
    x = synth.make_inputs(w, **make_kw)
    H = x.q.shape[1]
    g = Bd.Geometry(B=x.B, L=x.L, H=H, D=w.D, span=w.span, nb=w.nb, mp=w.mp, dropout_p=w.dropout_p, seed=11,
                    offset=0, fp32_fast=fp32_fast)
    if x.packed:
        g.cu_seqlens = x.cu_seqlens.to(dev)
        g.total_tokens = int(x.cu_seqlens[-1])
    if x.qmask is not None:
        g.query_mask, g.key_mask = x.qmask.to(dev), x.kmask.to(dev)
    q, k, v, qr, kr, do = [t.to(dev) for t in (x.q, x.k, x.v, x.qr, x.kr, x.dout)]
    g.band_bias = Bd.alloc_band_bias(g, q.dtype, dev)
    out = torch.empty_like(q)
    lse = torch.empty(g.lse_shape(), dtype=torch.float32, device=dev)
    grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(qr),
             torch.empty_like(kr))
    wsf = Bd.alloc_workspace(g, q.dtype, False, dev)
    wsb = Bd.alloc_workspace(g, q.dtype, True, dev)
    stream = torch.cuda.current_stream()
    fwd = lambda: Bd.attn_fwd(g, q, k, v, qr, kr, out=out, lse=lse, workspace=wsf)
    bwd = lambda: Bd.attn_bwd(g, q, k, v, qr, kr, out, lse, do, grads=grads, workspace=wsb)

    def both():
        fwd()
        bwd()

    res = {}
    for phase, fn in (("fwd", fwd), ("bwd", bwd), ("fwd_bwd", both)):
        fwd()   # the backward reads the forward's outputs
        for _ in range(warmup):
            flush.zero_()
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        res[phase] = quantiles([a.elapsed_time(b) for a, b in ev])
    if Bd.device_error(wsf) or Bd.device_error(wsb):
        raise SystemExit(f"device error word set while timing {name}")
    fl_f, fl_b = workload_flops(x, w, H)
    for phase, fl in (("fwd", fl_f), ("bwd", fl_b), ("fwd_bwd", fl_f + fl_b)):
        res[phase]["tflops_at_median"] = fl / (res[phase]["median"] * 1e-3) / 1e12
    shape = {"B": x.B, "L": x.L, "H": H, "D": w.D, "R": w.R,
             "dtype": "float32 (fast mode)" if fp32_fast else str(q.dtype).replace("torch.", ""),
             "dropout_p": w.dropout_p, "packed": x.packed, "masked": x.qmask is not None,
             "tokens": int(x.cu_seqlens[-1]), "fwd_flops": fl_f, "bwd_flops": fl_b}
    return {"shape": shape, **res}


def time_inference(dev, L, iters, warmup, flush, B=8, H=12):
    """Latency of the inference forward (df_attn_fwd_inference, no LSE) at a
    short length with the v3-base head layout and padding masks."""
    import torch

    from exact_deberta_disentangled_gb300 import binding as Bd
    from exact_deberta_disentangled_gb300 import synth

    w = synth.WORKLOADS["v3_base"]
    x = synth.make_inputs(w, B=B, L=L, H=H)
    g = Bd.Geometry(B=B, L=L, H=H, D=w.D, span=w.span, nb=w.nb, mp=w.mp, query_mask=x.qmask.to(dev),
                    key_mask=x.kmask.to(dev))
    q, k, v, qr, kr = [t.to(dev) for t in (x.q, x.k, x.v, x.qr, x.kr)]
    out = torch.empty_like(q)
    ws = Bd.alloc_workspace(g, q.dtype, False, dev)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        Bd.attn_fwd_inference(g, q, k, v, qr, kr, out=out, workspace=ws)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        Bd.attn_fwd_inference(g, q, k, v, qr, kr, out=out, workspace=ws)
        b.record(stream)
    torch.cuda.synchronize()
    if Bd.device_error(ws):
        raise SystemExit(f"device error word set in the inference forward at L={L}")
    qs = quantiles([a.elapsed_time(b) * 1e3 for a, b in ev])   # microseconds
    return {"B": B, "L": L, "H": H, "D": w.D, "unit": "us", **qs}


def time_side_steps(dev, iters, warmup, flush):
    """The steps on either side of the attention at a DeBERTa-v3-base layer
    over the 16,384-token workload (hidden 768 = 12 x 64, R = 512): fused QKV
    projection forward / backward (GEMM TFLOP/s: 2 T C 3HD forward, twice that
    backward), relative projections forward / backward, and packing the
    varlen workload's padded batch (rows of 12 x 64 bf16)."""
    import torch

    from exact_deberta_disentangled_gb300 import binding as Bd
    from exact_deberta_disentangled_gb300 import synth

    g = torch.Generator().manual_seed(21)
    T, C, H, D, R = 16384, 768, 12, 64, 512
    mk = lambda shape, sc=1.0: (torch.randn(shape, generator=g) * sc).to(torch.bfloat16).to(dev)
    x, w, b, dqkv = mk((T, C)), mk((3, H * D, C), C ** -0.5), mk((3, H * D), 0.1), mk((3, T, H * D))
    rel, gamma, beta = mk((R, C)), mk((C,), 0.1), mk((C,), 0.1)
    dqr, dkr = mk((H, R, D)), mk((H, R, D))
    stream = torch.cuda.current_stream()
    qr, kr, rel_ln, stats = Bd.rel_proj_fwd(rel, gamma, beta, 1e-7, w, b, H, D)
    dw = torch.empty_like(w)

    def timed(fn):
        for _ in range(warmup):
            flush.zero_()
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        for a, e in ev:
            flush.zero_()
            a.record(stream)
            fn()
            e.record(stream)
        torch.cuda.synchronize()
        return quantiles([a.elapsed_time(e) for a, e in ev])

    res = {"qkv_fwd": timed(lambda: Bd.qkv_proj_fwd(x, w, b)),
           "qkv_bwd": timed(lambda: Bd.qkv_proj_bwd(x, w, dqkv, dw=dw)),
           "rel_fwd": timed(lambda: Bd.rel_proj_fwd(rel, gamma, beta, 1e-7, w, b, H, D)),
           "rel_bwd": timed(lambda: Bd.rel_proj_bwd(rel, gamma, rel_ln, stats, w, dqr, dkr, dw))}
    fl = 2.0 * T * C * 3 * H * D
    res["qkv_fwd"]["tflops_at_median"] = fl / (res["qkv_fwd"]["median"] * 1e-3) / 1e12
    res["qkv_bwd"]["tflops_at_median"] = 2 * fl / (res["qkv_bwd"]["median"] * 1e-3) / 1e12
    # packing: the varlen workload's sequences as a padded batch of their longest length
    v = synth.make_inputs(synth.WORKLOADS["varlen"])
    lens = (v.cu_seqlens[1:] - v.cu_seqlens[:-1])
    nb, Lmax = len(lens), int(lens.max())
    mask = (torch.arange(Lmax)[None, :] < lens[:, None]).to(torch.uint8).to(dev)
    padded = torch.randn((nb, Lmax, H, D), generator=g).to(torch.bfloat16).to(dev)
    pi = Bd.pack_info(mask)
    packed = Bd.pack_rows(padded, pi)
    res["pack_info"] = timed(lambda: Bd.pack_info(mask))
    res["pack_rows"] = timed(lambda: Bd.pack_rows(padded, pi))
    res["unpack_rows"] = timed(lambda: Bd.unpack_rows(packed, pi))
    res["pack_bytes"] = 2 * pi.total * H * D * 2
    res["shapes"] = {"T": T, "C": C, "H": H, "D": D, "R": R, "pack_batch": [nb, Lmax], "pack_tokens": pi.total}
    return res


def run_extras(dev, iters, warmup, flush):
    """The length sweep and the other workloads, each timed separately
    (fwd, bwd alone, fwd + bwd; min / p10 / median / p90), plus the
    inference latency at short lengths."""
    sweep = {}
    for L in (512, 1024, 2048, 4096, 8192):
        sweep[f"L{L}"] = time_phases(f"sweep_L{L}", dev, iters, warmup, flush)
    configs = {}
    for name in ("v3_base", "varlen", "hd128_dropout", "hd32_dropout", "mnli_fp16"):
        configs[name] = time_phases(name, dev, iters, warmup, flush)
    # fp32 tensors: the fast mode (fp16 tensor-core path) at the L = 8192 sweep shape
    configs["fast_fp32_L8192"] = time_phases("sweep_L8192", dev, iters, warmup, flush, fp32_fast=True,
                                             dtype="fp32")
    infer = {f"L{L}": time_inference(dev, L, iters, warmup, flush) for L in (64, 128, 384)}
    side = time_side_steps(dev, iters, warmup, flush)
    return {"sweep": sweep, "configs": configs, "inference_latency": infer, "steps_either_side": side,
            "method": "CUDA events on the launching stream per iteration, L2 flushed (512 MB write) before "
                      "each; bwd timed alone from the saved forward outputs"}


def run_profile_case(args, local_rank):
    """Small case for kernel profiling (ncu): one sequence of the L=8192
    workload (B=1, H=12, 8,192 tokens: the same tile mix as the timed
    workload at half its size; inputs + diagonal-sum buffers ~330 MB > L2).
    Runs warmup + steps fwd+bwd iterations without timing."""
    import torch

    from exact_deberta_disentangled_gb300 import binding as Bd
    from exact_deberta_disentangled_gb300 import synth

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS["sweep_L8192"]
    x = synth.make_inputs(w, B=1)
    g = Bd.Geometry(B=x.B, L=x.L, H=w.H, D=w.D, span=w.span, nb=w.nb, mp=w.mp)
    q, k, v, qr, kr, do = [t.to(dev) for t in (x.q, x.k, x.v, x.qr, x.kr, x.dout)]
    g.band_bias = Bd.alloc_band_bias(g, q.dtype, dev)
    out, lse, wsf = Bd.attn_fwd(g, q, k, v, qr, kr)
    grads, wsb = Bd.attn_bwd(g, q, k, v, qr, kr, out, lse, do)
    for _ in range(args.warmup + args.steps - 1):
        Bd.attn_fwd(g, q, k, v, qr, kr, out=out, lse=lse, workspace=wsf)
        Bd.attn_bwd(g, q, k, v, qr, kr, out, lse, do, grads=grads, workspace=wsb)
    torch.cuda.synchronize()
    ef, eb = Bd.device_error(wsf), Bd.device_error(wsb)
    if ef or eb:
        raise SystemExit(f"device error word: forward {ef}, backward {eb}")
    print("profile case done", flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--ref-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the length sweep, the other workloads and the inference latencies")
    ap.add_argument("--extra-iters", type=int, default=15)
    ap.add_argument("--profile-run", action="store_true",
                    help="run the small profiling case (L=8192, B=1) without timing")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.profile_run:
        run_profile_case(args, local_rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_gpu(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
