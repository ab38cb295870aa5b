#!/usr/bin/env python
"""Benchmark of the Periodic Row-wise Muon optimizer step on one GB300 (or N replicas).

Default workload: the 15B-class MMDiT parameter set (440 matrices, H = 3072, bf16 W and
G, fp32 M), the largest set that fits one GPU.  One bench step = one period of the
K = 3 schedule over the whole set: an NS5 refresh step followed by two RowNorm steps
(every row of the hot path: schedule, momentum, Newton-Schulz, RowNorm, scale,
apply).  The reported value is the mean optimizer-step time (period / 3).  Vanilla
Muon (K = 1, every step a refresh) is timed next, on the same buffers, under the
`vanilla` key.  Inputs (W, G, M) are synthetic, on the device before the timed region,
and larger than L2.  Newton-Schulz GEMM time and RowNorm time come from CUDA events
that the library records on its stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]
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

METRIC = "Muon optimizer step ms; NS5 TFLOP/s and RowNorm GB/s vs GB300 roofline"
# The largest parameter set that fits one GPU (W, G, M and the workspace about 182 GB).
DEFAULT_WORKLOAD = "mmdit-15b"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129e6
# DRAM bytes per ns_tc_kernel launch (read + write, averaged over the 15 launches of
# a refresh), from ncu dram__bytes_{read,write}.sum on a slice of the set with the
# same shape mix (whole MMDiT blocks), scaled by the matrix count of the full set.
# Valid only for the kernel sources it was measured on (hash below); otherwise the
# roofline reports null.
NS5_TRAFFIC = {"mmdit-15b": {"bytes_per_launch": 6.161e10, "sources": "bf84e40d372c8c13"}}
NS5_SOURCES = ["ns_tc.cu", "ns_common.cuh", "ptx.cuh", "common.cuh", "internal.h", "api.cu"]


def ns5_sources_hash():
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "matrix_aware_optimizer_muon_gb300", "csrc")
    for f in NS5_SOURCES:
        with open(os.path.join(d, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph per-branch timing")
    ap.add_argument("--scale-mode", default="adjusted_lr", choices=["adjusted_lr", "update_norm"],
                    help="update scale: 0.2*sqrt(max(A,B)) (Eq. 7, default) or 0.2/RMS(U) (Eq. 6)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--K", type=int, default=0,
                    help="override the schedule period K (1 = vanilla Muon: every step is a refresh)")
    ap.add_argument("--full-oracle", action="store_true",
                    help="reference arm: also time the oracle over every matrix of the set for one period")
    ap.add_argument("--no-vanilla", action="store_true", help="skip the vanilla Muon (K=1) side-by-side timing")
    ap.add_argument("--e2e-buckets", type=int, default=16,
                    help="e2e: buckets of consecutive matrices a step is streamed in (one library call each)")
    ap.add_argument("--e2e-slots", type=int, default=0,
                    help="e2e: device buffers for gradient buckets (uploads run up to slots - 1 buckets ahead); "
                         "0: as many as device memory holds, up to two steps' worth")
    ap.add_argument("--debug-flags", type=int, default=0,
                    help="library test-hook flags for A/B timing (for example 16: one-CTA Newton-Schulz tiles)")
    ap.add_argument("--matrices", type=int, default=0,
                    help="keep only the first N matrices of the set (small cases for profiling)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK), "fallback"


# ---------------------------------------------------------------------------
# analytic work
# ---------------------------------------------------------------------------
def ns5_flops(shapes):
    """Dense count 5*(4 n^2 m + 2 n^3) per matrix, n = min(A, B), m = max(A, B)."""
    return sum(5 * (4 * min(a, b) ** 2 * max(a, b) + 2 * min(a, b) ** 3) for a, b in shapes)


def ns5_flops_symmetric(shapes):
    """Symmetric-minimum count 5*(3 n^2 m + n^3) per matrix: the two symmetric products
    (X X^T and S S) counted over one triangle each, the update B X in full."""
    return sum(5 * (3 * min(a, b) ** 2 * max(a, b) + min(a, b) ** 3) for a, b in shapes)


def ns5_flops_executed(shapes):
    """FLOPs the tensor-core kernels issue: 128x256 output tiles with K padded to 64;
    for the two symmetric products only the tiles that touch the upper triangle
    (row blocks up to 2*tn+1 of each 256-column block)."""
    tot = 0
    for a, b in shapes:
        n, m = min(a, b), max(a, b)
        mt = -(-n // 128)
        sym = sum(min(2 * t + 2, mt) for t in range(-(-n // 256)))
        kn, km = 64 * -(-n // 64), 64 * -(-m // 64)
        tile = 2 * 128 * 256
        tot += 5 * tile * (sym * km + sym * kn + mt * -(-m // 256) * kn)
    return tot


def rownorm_bytes(shapes, wb, gb):
    """Algorithmic bytes of a RowNorm step: read G, read+write M (fp32), read+write W."""
    return sum(a * b * (gb + 8 + 2 * wb) for a, b in shapes)


def momentum_bytes(shapes, gb, xb):
    """Algorithmic bytes of a refresh step's momentum pass: read G, read+write M (fp32),
    write X~ (the Newton-Schulz input, xb bytes per element)."""
    return sum(a * b * (gb + 8 + xb) for a, b in shapes)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons, pw = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            try:
                pw.append(float(f[3]))
            except ValueError:
                pass
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "power_w": statistics.median(pw) if pw else None}


# ---------------------------------------------------------------------------
# distributed helpers (replicas: no data-path collective)
# ---------------------------------------------------------------------------
def dist_init(torch):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, None
    import torch.distributed as dist
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    dist.init_process_group(backend)
    return dist.get_rank(), dist.get_world_size(), dist


def max_over_ranks(torch, dist, x: float, device) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---------------------------------------------------------------------------
# oracle (CPU) timing on a bounded sample
# ---------------------------------------------------------------------------
def oracle_units(wl):
    """Units of the oracle sample: one matrix of each shape group on a refresh step and,
    when K > 1, on a RowNorm step.  Returns (group, rows, cols, count, refresh) tuples."""
    units = []
    for gi, ((a, b), cnt) in enumerate(wl.shape_groups()):
        units.append((gi, a, b, cnt, True))
        if wl.K > 1:
            units.append((gi, a, b, cnt, False))
    return units


def time_oracle_unit(wl, unit, seed=0):
    """Seconds of one fp64 oracle optimizer step on one matrix of the unit's shape (inputs
    are made before the clock starts)."""
    import numpy as np
    from oracle import muon_ref
    from synth import gradient_np, quantize_np, weight_init_np
    gi, a, b, _, refresh = unit
    W = quantize_np(weight_init_np(a, b, seed, gi), wl.w_dtype).astype(np.float64)
    M = np.zeros((a, b))
    G = quantize_np(gradient_np(a, b, wl.spike_scales, seed, gi, 0), wl.g_dtype)
    step = 0 if refresh else 1
    t0 = time.perf_counter()
    muon_ref.periodic_step(W, M, G, step, wl.K, wl.gamma, wl.mu, wl.eta, wl.lam, w_dtype=wl.w_dtype)
    return time.perf_counter() - t0


def oracle_extrapolate(wl, times):
    """ms per optimizer step of the whole set from per-unit seconds ({unit: [s, ...]}):
    sum over shape groups of count * (refresh + (K - 1) * RowNorm) / K."""
    per_group = {}
    for u, ts in times.items():
        gi, a, b, cnt, refresh = u
        d = per_group.setdefault(gi, {"shape": [a, b], "count": cnt})
        d["refresh_s" if refresh else "rownorm_s"] = statistics.mean(ts)
    total = 0.0
    detail = []
    for gi in sorted(per_group):
        d = per_group[gi]
        rn = d.get("rownorm_s", 0.0)
        total += d["count"] * (d["refresh_s"] + (wl.K - 1) * rn) / wl.K
        detail.append({"shape": d["shape"], "count": d["count"], "refresh_s": round(d["refresh_s"], 4),
                       "rownorm_s": round(rn, 4) if wl.K > 1 else None})
    return total * 1e3, detail


def oracle_sample_text(wl):
    return (f"one matrix per shape group ({len(wl.shape_groups())} groups), each timed on one refresh step"
            + (" and one RowNorm step" if wl.K > 1 else "")
            + f" of the fp64 oracle; extrapolated by group counts to the {len(wl.matrices)} matrices "
            f"and the K={wl.K} schedule")


def select_workload(args):
    import dataclasses
    from synth import WORKLOADS
    wl = WORKLOADS[args.workload]
    if args.matrices and args.matrices < len(wl.matrices):
        wl = dataclasses.replace(wl, key=f"{wl.key}[:{args.matrices}]", matrices=wl.matrices[:args.matrices])
    if args.K and args.K != wl.K:
        wl = dataclasses.replace(wl, key=f"{wl.key}/K={args.K}", K=args.K)
    return wl


def config_dict(wl, args, world):
    """The workload description both arms print (the same keys and values)."""
    shapes = [(m.rows, m.cols) for m in wl.matrices]
    wb = 2 if wl.w_dtype == "bf16" else 4
    gb = 2 if wl.g_dtype == "bf16" else 4
    in_bytes = sum(-(-(a * b) // 128) * 128 for a, b in shapes) * (wb + gb + 4)
    flush = in_bytes < 4 * L2_BYTES
    return {"workload": wl.key, "matrices": len(shapes), "params": wl.n_params,
            "K": wl.K, "gamma": wl.gamma, "mu": wl.mu, "eta": wl.eta, "lambda": wl.lam,
            "scale_mode": args.scale_mode,
            "step": (f"one K={wl.K} period: 1 NS5 refresh + {wl.K - 1} RowNorm optimizer steps; value = period/{wl.K}"
                     if wl.K > 1 else "vanilla Muon (K=1): every optimizer step is an NS5 refresh"),
            "l2": (f"inputs larger than L2 (W+G+M {in_bytes / 1e9:.1f} GB vs 129 MB L2), no flush" if not flush
                   else f"inputs fit in L2 ({in_bytes / 1e6:.1f} MB): L2 flushed (256 MB write) before every "
                        "timed period; period timed by the library's phase events, excluding the flush"),
            "parallelism": "replicas" if world > 1 else "single GPU"}, in_bytes, flush


def run_reference(args, torch):
    """The fp64 oracle on the host cores.  One bench step times one unit of the sample
    (one matrix of one shape group on one branch), in round-robin order over the units;
    the value extrapolates the per-unit means to the whole set.  Units that --steps does
    not reach are timed once more after the timed steps, so that every group counts."""
    rank, world, dist = dist_init(torch)
    if rank != 0:
        return
    wl = select_workload(args)
    units = oracle_units(wl)
    cheapest = min(units, key=lambda u: (u[4], u[1] * u[2]))
    for _ in range(min(args.warmup, 1)):   # the oracle needs no more warm-up than one import and one call
        time_oracle_unit(wl, cheapest)
    times = {u: [] for u in units}
    wall0 = time.perf_counter()
    for i in range(args.steps):
        u = units[i % len(units)]
        times[u].append(time_oracle_unit(wl, u))
    wall = time.perf_counter() - wall0
    step_s = [t for ts in times.values() for t in ts]
    extra = [u for u in units if not times[u]]
    for u in extra:
        times[u].append(time_oracle_unit(wl, u))
    value, detail = oracle_extrapolate(wl, times)
    cfg, _, _ = config_dict(wl, args, 1)
    sample = oracle_sample_text(wl) + (f"; bench step i times unit i mod {len(units)}"
                                       + (f"; {len(extra)} units beyond --steps timed once more" if extra else ""))
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "ms", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(statistics.mean(step_s) * 1e3, 3) if step_s else None,
            "ms_per_step_is": "measured wall time of one bench step (one unit of the sample)",
            "extrapolated_ms_per_period": round(value * wl.K, 3),
            "wall_s_timed_steps": round(wall, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": round(value, 3), "unit": "ms", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample, "detail": detail},
            "e2e": {"value": round(value, 3), "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    if args.full_oracle:
        line["full_oracle"] = full_oracle_period(wl)
    print(json.dumps(line), flush=True)


def full_oracle_period(wl, seed=0):
    """The fp64 oracle over every matrix of the set through one K-step period (no
    extrapolation): ms per optimizer step."""
    import numpy as np
    from oracle import muon_ref
    from synth import gradient_np, quantize_np, weight_init_np
    tot = 0.0
    for i, m in enumerate(wl.matrices):
        a, b = m.rows, m.cols
        W = quantize_np(weight_init_np(a, b, seed, i), wl.w_dtype).astype(np.float64)
        M = np.zeros((a, b))
        for step in range(wl.K):
            G = quantize_np(gradient_np(a, b, wl.spike_scales, seed, i, step), wl.g_dtype)
            t0 = time.perf_counter()
            W, M, _ = muon_ref.periodic_step(W, M, G, step, wl.K, wl.gamma, wl.mu, wl.eta, wl.lam,
                                             w_dtype=wl.w_dtype)
            tot += time.perf_counter() - t0
    return {"value": round(tot * 1e3 / wl.K, 3), "unit": "ms", "cores": os.cpu_count(),
            "sample": f"all {len(wl.matrices)} matrices through one K={wl.K} period, timed step by step"}


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------
def e2e_buckets(offs, tot, nb):
    """Split the matrix list into at most nb runs of consecutive matrices holding about
    equal bytes: [(first matrix, end matrix, first element, end element)]."""
    ends = offs[1:] + [tot]
    cuts, k = [0], 1
    for j, e in enumerate(ends):
        if k < nb and e >= tot * k / nb and j + 1 < len(offs):
            cuts.append(j + 1)
            while k < nb and e >= tot * k / nb:
                k += 1
    cuts.append(len(offs))
    return [(a, b, offs[a], ends[b - 1]) for a, b in zip(cuts, cuts[1:]) if b > a]


def run_e2e(args, torch, mm, dist, device, wl, shapes, offs, tot, W_flat, G_flat, W, M, ws, mode, step_counter,
            gdt, wdt, gb, wb):
    """The optimizer step end to end through the public call: every step uploads its
    gradients from pinned host memory and downloads the updated weights to pinned host
    memory, both inside the timed region.  The matrices are taken in buckets of
    consecutive matrices (one muon_periodic_step call each), the way a training loop
    would stream them, so that bucket b's copies overlap the other buckets' compute."""
    buckets = e2e_buckets(offs, tot, max(1, args.e2e_buckets))
    span = max(e - s for (_, _, s, e) in buckets)
    torch.cuda.empty_cache()
    free = torch.cuda.mem_get_info(device)[0]
    # G slots: a ring of device buffers of one bucket each, so that uploads run up to
    # nslot - 1 buckets ahead of the compute.  A refresh step computes for about as long
    # as two steps' copies take, so the uploads of the following steps must be able to
    # run that far ahead of it: by default as many slots as fit, up to two steps' worth.
    want = args.e2e_slots if args.e2e_slots > 0 else 2 * len(buckets) + 1
    nslot = 0
    for k in range(want, 0, -1):
        if k * span * gb + (2 << 30) <= free:
            nslot = k
            break
    if nslot == 0:
        return {"value": None, "unit": "ms",
                "skipped": f"not enough device memory for one gradient bucket ({free / 1e9:.1f} GB free, "
                           f"{(span * gb + (2 << 30)) / 1e9:.1f} GB needed)"}
    # pinned host copies of G and W (60 GB per rank at 15B): several replicas on one
    # node may not find that much page-locked memory; then the leg reports why
    try:
        G_host = torch.empty(tot, dtype=gdt, pin_memory=True)
        W_host = torch.empty(tot, dtype=wdt, pin_memory=True)
    except RuntimeError as exc:
        return {"value": None, "unit": "ms", "skipped": f"pinned host buffers not available: {str(exc)[:160]}"}
    G_host.copy_(G_flat)
    slots = [torch.empty(span, dtype=gdt, device=device) for _ in range(nslot)]
    views = [[[sl[offs[j] - s0:offs[j] - s0 + shapes[j][0] * shapes[j][1]].view(*shapes[j]) for j in range(a, b)]
              for (a, b, s0, _) in buckets] for sl in slots]
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    nb = len(buckets)
    n_e2e = max(1, args.steps) * wl.K   # the device-timed region's optimizer steps
    items = n_e2e * nb                  # item q: step q // nb, bucket q % nb
    uploaded = [torch.cuda.Event() for _ in range(nslot)]
    consumed = [torch.cuda.Event() for _ in range(nslot)]
    updated = [torch.cuda.Event() for _ in range(nb)]
    downloaded = [torch.cuda.Event() for _ in range(nb)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def upload(q):   # item q's gradients into slot q % nslot, once item q - nslot has read that slot
        a, b, s0, s1 = buckets[q % nb]
        with torch.cuda.stream(up):
            if q >= nslot:
                up.wait_event(consumed[q % nslot])
            slots[q % nslot][:s1 - s0].copy_(G_host[s0:s1], non_blocking=True)
            uploaded[q % nslot].record(up)

    def download(q):   # bucket q % nb's updated weights to the host
        a, b, s0, s1 = buckets[q % nb]
        with torch.cuda.stream(down):
            down.wait_event(updated[q % nb])
            W_host[s0:s1].copy_(W_flat[s0:s1], non_blocking=True)
            downloaded[q % nb].record(down)

    barrier(dist)
    e0.record(comp)
    up.wait_event(e0)
    down.wait_event(e0)
    for q in range(min(nslot - 1, items)):
        upload(q)
    for q in range(items):
        if q + nslot - 1 < items:
            upload(q + nslot - 1)
        i, bk = divmod(q, nb)
        a, b, _, _ = buckets[bk]
        comp.wait_event(uploaded[q % nslot])
        if i >= 1:   # the previous step's download of these weights must have read them
            comp.wait_event(downloaded[bk])
        mm.muon_periodic_step(W[a:b], views[q % nslot][bk], M[a:b], step_counter[0] + i, ws, K=wl.K,
                              gamma=wl.gamma, mu=wl.mu, eta=wl.eta, lam=wl.lam, ns5_mode=mode,
                              scale_mode=args.scale_mode)
        consumed[q % nslot].record(comp)
        updated[bk].record(comp)
        download(q)
    comp.wait_stream(down)
    e1.record(comp)
    torch.cuda.synchronize()
    step_counter[0] += n_e2e
    if mm.muon_check_status(ws) != mm.MUON_OK:
        raise RuntimeError("device status error in the end-to-end run")
    e2e_ms = max_over_ranks(torch, dist, e0.elapsed_time(e1) / n_e2e, device)
    # The same copies with no compute between them: the floor the host link sets.
    l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0.record(comp)
    for s_, is_up in ((up, True), (down, False)):
        with torch.cuda.stream(s_):
            s_.wait_event(l0)
            for q in range(items):
                a, b, s0, s1 = buckets[q % nb]
                if is_up:
                    slots[q % nslot][:s1 - s0].copy_(G_host[s0:s1], non_blocking=True)
                else:
                    W_host[s0:s1].copy_(W_flat[s0:s1], non_blocking=True)
        comp.wait_stream(s_)
    l1.record(comp)
    torch.cuda.synchronize()
    link_ms = max_over_ranks(torch, dist, l0.elapsed_time(l1) / n_e2e, device)
    return {"value": round(e2e_ms, 4), "unit": "ms", "h2d_bytes_per_step": tot * gb,
            "d2h_bytes_per_step": tot * wb, "steps": n_e2e,
            "copies_alone_ms": round(link_ms, 4),
            "copies_alone_gbs": round((tot * gb + tot * wb) / link_ms / 1e6, 1),
            "buckets": nb, "gradient_slots": nslot,
            "note": "every step: G uploaded from and W downloaded to pinned host memory, "
                    f"in {nb} buckets of consecutive matrices (one muon_periodic_step call each; "
                    f"{nslot} device slots for G buckets, so uploads run ahead of the compute; "
                    "a bucket's download overlaps the next buckets' compute); the timed region "
                    "holds one pipeline fill (first upload) and drain (last download); "
                    "copies_alone_ms: the same copies with no compute"}


def run_ours(args, torch):
    import matrix_aware_optimizer_muon_gb300 as mm
    from synth import WORKLOADS, gradient_torch, weight_init_torch

    rank, world, dist = dist_init(torch)
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    mm.load_library()
    if args.debug_flags:
        mm.muon_debug_set(args.debug_flags, 0)
    wl = select_workload(args)
    shapes = [(m.rows, m.cols) for m in wl.matrices]
    wdt = torch.bfloat16 if wl.w_dtype == "bf16" else torch.float32
    gdt = torch.bfloat16 if wl.g_dtype == "bf16" else torch.float32
    wb, gb = (2 if wl.w_dtype == "bf16" else 4), (2 if wl.g_dtype == "bf16" else 4)

    # flat device buffers (one H2D / D2H copy each for the end-to-end run)
    offs, tot = [], 0
    for a, b in shapes:
        offs.append(tot)
        tot += -(-(a * b) // 128) * 128
    W_flat = torch.empty(tot, dtype=wdt, device=device)
    G_flat = torch.empty(tot, dtype=gdt, device=device)
    M_flat = torch.zeros(tot, dtype=torch.float32, device=device)
    W = [W_flat[o:o + a * b].view(a, b) for o, (a, b) in zip(offs, shapes)]
    G = [G_flat[o:o + a * b].view(a, b) for o, (a, b) in zip(offs, shapes)]
    M = [M_flat[o:o + a * b].view(a, b) for o, (a, b) in zip(offs, shapes)]
    seed = 1234 + rank
    for i, (a, b) in enumerate(shapes):
        W[i].copy_(weight_init_torch(torch, device, a, b, seed, i, wdt))
        gradient_torch(torch, device, a, b, wl.spike_scales, seed, i, 0, gdt, out=G[i])
    ws = mm.alloc_workspace(shapes, "bf16" if wl.w_dtype == "bf16" else "f32", device=device)
    mode = "bf16" if wl.w_dtype == "bf16" else "f32"
    stream = torch.cuda.current_stream()

    launches = [0]

    def opt_step(step):
        mm.muon_periodic_step(W, G, M, step, ws, K=wl.K, gamma=wl.gamma, mu=wl.mu, eta=wl.eta, lam=wl.lam,
                              ns5_mode=mode, scale_mode=args.scale_mode)
        launches[0] += mm.muon_launch_count()

    step_counter = [0]

    def period(evsets=None):
        for _ in range(wl.K):
            if evsets is not None:
                mm.muon_profile_events(evsets)
            opt_step(step_counter[0])
            step_counter[0] += 1

    # warm-up (also the first call configures the kernels)
    for _ in range(args.warmup):
        period()
    torch.cuda.synchronize()
    if mm.muon_check_status(ws) != mm.MUON_OK:
        raise RuntimeError("device status error during warm-up")

    # timed region: per-period event sets record the phase boundaries
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    for s in evs:
        for e in s:
            e.record()
    t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # Sets whose inputs fit in L2 get an L2 flush (a 256 MB write) before every timed
    # period; their period time then comes from the library's own phase events, which
    # exclude the flush.
    cfg, in_bytes, flush = config_dict(wl, args, world)
    scratch = torch.empty(64 << 20, dtype=torch.float32, device=device) if flush else None
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(dist)
    torch.cuda.synchronize()
    launches[0] = 0
    wall0 = time.perf_counter()
    t0e.record()
    for i in range(args.steps):
        if flush:
            scratch.fill_(float(i))
        period(evs[i])
    t1e.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(dist)
    clk = clocks.stop()
    mm.muon_profile_events([])
    if mm.muon_check_status(ws) != mm.MUON_OK:
        raise RuntimeError("device status error in the timed region")
    if flush:   # refresh start to the end of the period's last step, per period
        period_ms = statistics.mean(s[0].elapsed_time(s[4] if wl.K > 1 else s[2]) for s in evs)
    else:
        period_ms = t0e.elapsed_time(t1e) / args.steps
    period_ms = max_over_ranks(torch, dist, period_ms, device)
    refresh_ms = statistics.mean(s[0].elapsed_time(s[2]) for s in evs)
    ns5_ms = statistics.mean(s[1].elapsed_time(s[2]) for s in evs)
    mom_ms = statistics.mean(s[0].elapsed_time(s[1]) for s in evs)   # momentum + ||M|| + X~ pass
    has_rn = wl.K > 1   # K = 1 (vanilla Muon) has no RowNorm steps
    rownorm_ms = statistics.mean(s[3].elapsed_time(s[4]) for s in evs) if has_rn else None   # last RowNorm step of each period
    gpu_launches = launches[0] // args.steps

    flops = ns5_flops(shapes)
    flops_sym = ns5_flops_symmetric(shapes)
    flops_exec = ns5_flops_executed(shapes)
    rn_bytes = rownorm_bytes(shapes, wb, gb)
    pk, pk_src = peaks()
    ns5_tflops = flops / (ns5_ms * 1e-3) / 1e12
    ns5_sym_tflops = flops_sym / (ns5_ms * 1e-3) / 1e12
    ns5_exec_tflops = flops_exec / (ns5_ms * 1e-3) / 1e12
    rn_gbs = rn_bytes / (rownorm_ms * 1e-3) / 1e9 if has_rn else None
    mom_bytes = momentum_bytes(shapes, gb, 2 if mode == "bf16" else 4)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    fp32_peak = sms * 128 * 2 * ((clk or {}).get("sm_max_mhz") or 2070.0) * 1e6 / 1e12
    mom_gbs = mom_bytes / (mom_ms * 1e-3) / 1e9
    peak_tc = pk.get("bf16_tflops_sustained", FALLBACK["bf16_tflops_sustained"])
    peak_hbm = pk.get("hbm_gbs", FALLBACK["hbm_gbs"])
    n_ns5_launches = 15 * max(1, math.ceil(len(wl.shape_groups()) / 8))
    tr = NS5_TRAFFIC.get(wl.key)
    ns5_traffic = tr["bytes_per_launch"] if tr and tr["sources"] == ns5_sources_hash() else None

    line = {
        "metric": METRIC, "value": round(period_ms / wl.K, 4), "unit": "ms", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(period_ms, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if mode == "bf16" else "f32",
        "data": "synthetic",
        "config": cfg,
        "refresh_ms": round(refresh_ms, 4), "ns5_ms": round(ns5_ms, 4),
        "rownorm_ms": round(rownorm_ms, 4) if has_rn else None,
        "ns5_tflops": round(ns5_sym_tflops, 1), "ns5_tflops_dense": round(ns5_tflops, 1),
        "ns5_tflops_executed": round(ns5_exec_tflops, 1),
        "rownorm_gbs": round(rn_gbs, 1) if has_rn else None,
        "roofline": ({"kernel": "ns_tc_kernel (Newton-Schulz GEMMs)", "bound": "tensor",
                      "achieved": round(ns5_sym_tflops, 1), "peak": peak_tc, "unit": "TFLOP/s",
                      "frac": round(ns5_sym_tflops / peak_tc, 4), "traffic": ns5_traffic,
                      "work": "symmetric-minimum count 5*(3 n^2 m + n^3) per matrix (n = min(A,B), m = max(A,B))",
                      "flops_per_refresh": flops_sym, "launches_per_refresh": n_ns5_launches,
                      "achieved_dense": round(ns5_tflops, 1), "frac_dense": round(ns5_tflops / peak_tc, 4),
                      "flops_dense_per_refresh": flops,
                      "achieved_executed": round(ns5_exec_tflops, 1),
                      "frac_executed": round(ns5_exec_tflops / peak_tc, 4),
                      "peak_source": f"{pk_src} bf16_tflops_sustained",
                      "frac_of_nominal_2250": round(ns5_sym_tflops / 2250.0, 4)} if mode == "bf16" else
                     {"kernel": "ns_simt_kernel (fp32 Newton-Schulz GEMMs on the CUDA cores)", "bound": "alu",
                      "achieved": round(ns5_tflops, 2), "peak": round(fp32_peak, 1), "unit": "TFLOP/s",
                      "frac": round(ns5_tflops / fp32_peak, 4), "traffic": None,
                      "peak_source": "derived: SMs x 128 FFMA/clk x 2 FLOP x max SM clock",
                      "flops_per_refresh": flops}),
        "momentum_ms": round(mom_ms, 4), "momentum_gbs": round(mom_gbs, 1),
        "momentum_roofline": {"bound": "hbm", "achieved": round(mom_gbs, 1), "peak": peak_hbm, "unit": "GB/s",
                              "frac": round(mom_gbs / peak_hbm, 4), "bytes_per_refresh": mom_bytes,
                              "what": "refresh step's momentum pass: M <- mu*M + G, ||M||_F partials, X~ for NS5",
                              "peak_source": f"{pk_src} hbm_gbs"},
        "rownorm_roofline": {"bound": "hbm", "achieved": round(rn_gbs, 1), "peak": peak_hbm, "unit": "GB/s",
                             "frac": round(rn_gbs / peak_hbm, 4), "bytes_per_step": rn_bytes,
                             "peak_source": f"{pk_src} hbm_gbs", "frac_of_nominal_8000": round(rn_gbs / 8000.0, 4)}
        if has_rn else None,
        "gpu_launches": gpu_launches,
        "clocks": clk,
        "wall_s": round(wall, 3),
    }
    if args.debug_flags:
        line["debug_flags"] = args.debug_flags

    # Vanilla Muon (K = 1: every optimizer step an NS5 refresh) on the same buffers,
    # timed right after the periodic schedule, as the pages compare the two.
    if wl.K > 1 and not args.no_vanilla:
        n_v = max(1, args.steps)

        def vstep():
            mm.muon_periodic_step(W, G, M, step_counter[0], ws, K=1, gamma=wl.gamma, mu=wl.mu, eta=wl.eta,
                                  lam=wl.lam, ns5_mode=mode, scale_mode=args.scale_mode)
            step_counter[0] += 1

        for _ in range(max(1, min(args.warmup, 3))):
            vstep()
        vevs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_v)]
        for s_ in vevs:
            for e in s_:
                e.record()
        v0, v1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        vclocks = ClockSampler(local)
        vclocks.start()
        time.sleep(0.3)
        barrier(dist)
        torch.cuda.synchronize()
        v0.record()
        for i in range(n_v):
            mm.muon_profile_events(vevs[i])
            vstep()
        v1.record()
        torch.cuda.synchronize()
        barrier(dist)
        vclk = vclocks.stop()
        mm.muon_profile_events([])
        if mm.muon_check_status(ws) != mm.MUON_OK:
            raise RuntimeError("device status error in the vanilla Muon steps")
        v_ms = max_over_ranks(torch, dist, v0.elapsed_time(v1) / n_v, device)
        v_ns5 = statistics.mean(s_[1].elapsed_time(s_[2]) for s_ in vevs)
        line["vanilla"] = {
            "what": "vanilla Muon (K=1, every step an NS5 refresh) on the same buffers, timed after the "
                    f"K={wl.K} schedule",
            "ms_per_step": round(v_ms, 4), "steps": n_v, "warmup": max(1, min(args.warmup, 3)),
            "ns5_ms": round(v_ns5, 4), "ns5_tflops": round(flops_sym / (v_ns5 * 1e-3) / 1e12, 1),
            "periodic_ms_per_step": line["value"],
            "optimizer_time_cut": round(1.0 - line["value"] / v_ms, 4),
            "clocks": vclk}

    # Per-branch timing as CUDA-graph replays: one refresh step and one RowNorm step are
    # each captured once and replayed 20 times (the median of the per-replay event
    # times is reported).  Replays repeat the same step on the same buffers, which is
    # what a timing of the step needs; the schedule itself was exercised above.
    if not args.no_graph:
        try:
            gstream = torch.cuda.Stream()
            gstream.wait_stream(torch.cuda.current_stream())
            graphs = {}
            branches = [("refresh", 0)] + ([("rownorm", 1)] if wl.K > 1 else [])
            with torch.cuda.stream(gstream):
                for name, st in branches:   # warm the exact call once on this stream
                    mm.muon_periodic_step(W, G, M, st, ws, K=wl.K, gamma=wl.gamma, mu=wl.mu, eta=wl.eta,
                                          lam=wl.lam, ns5_mode=mode, scale_mode=args.scale_mode)
            torch.cuda.synchronize()
            for name, st in branches:
                g_ = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g_, stream=gstream):
                    mm.muon_periodic_step(W, G, M, st, ws, K=wl.K, gamma=wl.gamma, mu=wl.mu, eta=wl.eta,
                                          lam=wl.lam, ns5_mode=mode, scale_mode=args.scale_mode)
                graphs[name] = g_
            torch.cuda.synchronize()
            gres = {}
            for name, g_ in graphs.items():
                g_.replay()
                torch.cuda.synchronize()
                ts = []
                for _ in range(20):
                    if flush:
                        scratch.fill_(0.0)
                    a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a_.record()
                    g_.replay()
                    b_.record()
                    torch.cuda.synchronize()
                    ts.append(a_.elapsed_time(b_))
                gres[name + "_ms_median"] = round(statistics.median(ts), 4)
            if mm.muon_check_status(ws) != mm.MUON_OK:
                raise RuntimeError("device status error in the graph replays")
            if wl.K > 1:
                gres["k_average_ms"] = round((gres["refresh_ms_median"] + (wl.K - 1) * gres["rownorm_ms_median"])
                                             / wl.K, 4)
            gres["replays"] = 20
            line["graph"] = gres
        except RuntimeError as exc:   # capture unsupported here: leave the field out, say why
            line["graph"] = {"skipped": str(exc)[:200]}

    if not args.no_e2e:
        line["e2e"] = run_e2e(args, torch, mm, dist, device, wl, shapes, offs, tot, W_flat, G_flat, W, M, ws, mode,
                              step_counter, gdt, wdt, gb, wb)

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t0c = time.perf_counter()
        v, detail = oracle_extrapolate(wl, {u: [time_oracle_unit(wl, u)] for u in oracle_units(wl)})
        line["cpu_baseline"] = {"value": round(v, 3), "unit": "ms", "cores": os.cpu_count(), "kind": "oracle",
                                "sample": oracle_sample_text(wl) + " (each unit timed once)",
                                "cpu_s": round(time.perf_counter() - t0c, 1), "detail": detail}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    args = parse()
    import torch
    if args.impl == "reference":
        run_reference(args, torch)
    else:
        run_ours(args, torch)


if __name__ == "__main__":
    main()
