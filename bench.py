#!/usr/bin/env python
"""Benchmark one DSV sparse-attention layer step on GB300.

A step is one pass of the whole hot path over one batch of synthetic input, for every head
of the layer: low-rank estimate + top-k per query block -> sparse attention forward ->
sparse attention backward (dQ, dK, dV), all through the C ABI (libdsv.so).  The default
workload is the long video: 24 heads of N = 520,192 tokens at d = 128, k = 52,019 (10 %),
run as 6 calls of 4 heads (the selection of 4 heads takes 6.8 GB).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload long] [--impl dsv|reference]

Prints ONE JSON line (rank 0).  `value` is the effective TFLOP/s of the whole job:
14 * B * H * N * k * d flops per step (4 N k d forward + 10 N k d backward, only the
selected query-key pairs counted) divided by the step time, which includes the
estimate/top-k.  Inputs are resident in HBM when the timed region starts (drawn there by a
seeded device generator); between timed steps (outside the timed events) a 512 MiB memset
flushes L2 and a read of another 512 MiB buffer leaves it holding clean lines.  `e2e` is the
same metric when every head group's inputs are also copied host->device from pinned memory
and its outputs (O, LSE, dQ, dK, dV) back, inside the timed region.  Under torchrun each rank
runs an independent replica (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

REPO = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, REPO)

METRIC = "sparse attn fwd+bwd effective TFLOP/s and tokens/s at 10% density; % of bf16 peak"
CSRC = os.path.join(REPO, "dynamic_sparse_attention_estimate_gb300", "csrc")
TRAFFIC_FILE = os.path.join(REPO, "profiles", "kernel_traffic.json")
GIB = 1 << 30


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="long", help="tiny, short, mid, sweep or long (default: long)")
    ap.add_argument("--density", type=float, default=None)
    ap.add_argument("--impl", default="dsv", choices=["dsv", "reference"])
    ap.add_argument("--heads", type=int, default=None,
                    help="run the workload with this many heads (small cases for profiler captures)")
    ap.add_argument("--ws-gib", type=float, default=64.0,
                    help="backward workspace cap in GiB when a head group's partial rows do not fit one wave")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-adaptive", action="store_true", help="skip the mass-based selection measurement")
    ap.add_argument("--no-adaln", action="store_true", help="skip the fused AdaLN measurement")
    ap.add_argument("--no-side", action="store_true", help="skip every side measurement (dense, adaptive, AdaLN)")
    ap.add_argument("--profile-once", action="store_true",
                    help="run the first head group's estimate, forward and backward once, in the launch "
                         "configuration the timed step uses, and exit (for profiler captures)")
    return ap.parse_args(argv)


def workload(args):
    from dynamic_sparse_attention_estimate_gb300.inputs import WORKLOADS
    wl = WORKLOADS[args.workload]
    if args.density is not None:
        wl = wl.with_density(args.density)
    if args.heads is not None:
        wl = wl.with_heads(args.heads)
    return wl


def heads_per_call(wl):
    """Heads per library call: the long clip runs its heads 4 at a time (its idx for 4 heads is
    6.8 GB); the other workloads run all heads in one call."""
    return min(wl.heads_per_call or wl.H, wl.H)


def config_of(wl):
    t, h, w = wl.latent
    hpc = heads_per_call(wl)
    calls = (wl.H + hpc - 1) // hpc
    per_call = f" ({calls} calls of {hpc} heads)" if calls > 1 else ""
    return {"workload": f"{wl.name}: B={wl.B} H={wl.H}{per_call} latent {t}x{h}x{w} -> N={wl.N}, d={wl.d}, "
                        f"r={wl.r}, k={wl.k} ({100 * wl.density:.1f}% density), query blocks of 64",
            "B": wl.B, "H": wl.H, "heads_per_call": hpc, "N": wl.N, "d": wl.d, "r": wl.r, "k": wl.k, "block": 64,
            "density": round(wl.density, 4),
            "l2": "flushed between timed steps (outside the timed events): 512 MiB memset, then a read of another "
                  "512 MiB; a step's inputs (%.1f GB) %s L2" % (step_input_bytes(wl) / 1e9,
                                                              "exceed" if step_input_bytes(wl) > 129e6 else "fit in")}


def step_input_bytes(wl):
    return wl.B * wl.H * wl.N * (4 * wl.d + 2 * wl.r) * 2


def flops_per_step(wl):
    return 14.0 * wl.B * wl.H * wl.N * wl.k * wl.d


# ---------------------------------------------------------------- CPU oracle (baseline and reference arm)

def oracle_sample(wl, budget_s, cache={}):
    """Run the fp64 oracle (estimate, forward, backward) on consecutive query blocks of
    head 0 for about budget_s seconds.  Returns (effective flops done, seconds, blocks)."""
    import numpy as np
    import oracle
    from dynamic_sparse_attention_estimate_gb300.inputs import make_head
    key = (wl.name, wl.k, wl.N)
    if key not in cache:
        x = make_head(wl, 0, 0)
        cache[key] = ({k: v.float().numpy().astype(np.float64) for k, v in x.items()}, [0])
    f, nxt = cache[key]
    t0 = time.perf_counter()
    nblocks = 0
    while nblocks == 0 or time.perf_counter() - t0 < budget_s:
        b = nxt[0] % wl.NB
        nxt[0] += 1
        idx = oracle.estimate_topk(f["q_lr"], f["k_lr"], 64, wl.k, blocks=[b])
        full_idx = np.zeros((wl.NB, wl.k), np.int32)
        full_idx[b] = idx[0]
        o, lse = oracle.sparse_attn_fwd(f["q"], f["k"], f["v"], full_idx, 64, blocks=[b])
        oracle.sparse_attn_bwd(f["do"], f["q"], f["k"], f["v"], full_idx, 64, blocks=[b], o=o, lse=lse)
        nblocks += 1
    dt = time.perf_counter() - t0
    return 14.0 * 64 * nblocks * wl.k * wl.d, dt, nblocks


def dsv_sparse_attn_bwd_csr_workspace_bytes(wl, pairs, H=None):
    from dynamic_sparse_attention_estimate_gb300.binding import dsv_sparse_attn_bwd_csr_workspace, make_dims
    return dsv_sparse_attn_bwd_csr_workspace(make_dims(wl.B, H or wl.H, wl.N, wl.d, wl.r, wl.k), pairs)


def max_over_ranks(ms, dev, world):
    """The slowest rank's time (the job is done when every rank is); identity for one rank."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, steps, flop_per_rank_step, ms):
    """Whole-job throughput: every rank's work over the slowest rank's time (weak scaling)."""
    return world * steps * flop_per_rank_step / (ms / 1e3) / 1e12


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    wl = workload(args)
    per_step = max(0.05, 120.0 / max(1, args.steps + args.warmup))   # whole run about two minutes
    for _ in range(args.warmup):
        oracle_sample(wl, per_step)
    flops, secs, blocks = 0.0, 0.0, 0
    for _ in range(args.steps):
        fl, dt, nb = oracle_sample(wl, per_step)
        flops += fl
        secs += dt
        blocks += nb
    value = flops / secs / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(wl),
            "step": "estimate, forward and backward of sampled query blocks by the fp64 oracle on the host cores",
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"{blocks} query blocks of head 0 (estimate + forward + backward), "
                                       f"~{per_step:.2f} s per step, numpy fp64"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.index), "-lms", "50"], stdout=self.file,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t_start, t_end):
        self.file.flush()
        rows = []
        try:
            with open(self.file.name) as fh:
                for line in fh:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 9 or not parts[1].replace(".", "").isdigit():
                        continue
                    try:
                        ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    except ValueError:
                        ts = None
                    if ts is None or t_start - 0.05 <= ts <= t_end + 0.05:
                        rows.append(parts)
        finally:
            os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        mx = max(float(r[2]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        powers = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": reasons, "samples": len(rows),
                "power_w_max": max(powers) if powers else None}


# ---------------------------------------------------------------- roofline bookkeeping

def measured_peaks():
    p = os.path.join(REPO, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


KERNEL_FILES = {"estimate_topk": ("dsv_estimate.cu",), "estimate_arange": ("dsv_estimate.cu",),
                "sparse_fwd": ("dsv_fwd_tc.cu", "dsv_tc.cuh"), "bwd_main": ("dsv_bwd_tc.cu", "dsv_tc.cuh")}


def kernel_source_hash(kernel):
    """Hash of the sources a kernel is built from: stored DRAM traffic counts only while it matches."""
    h = hashlib.sha256()
    for f in KERNEL_FILES.get(kernel, ("dsv_bwd.cu",)) + ("dsv_common.cuh", "dsv_internal.h"):
        for ln in open(os.path.join(CSRC, f), encoding="utf-8"):
            code = ln.split("//", 1)[0].rstrip()  # comments do not change the kernel
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def algorithmic(kernel, wl, launches_per_step):
    """(bound, amount per launch, unit) for a kernel of the step: flops of the selected pairs for the
    attention kernels; for the HBM-bound kernels the bytes they must move (the reduce: every bf16
    partial row and its list entry read, dK and dV written)."""
    BH = wl.B * wl.H
    pairs = BH * wl.NB * wl.k
    dense = wl.k == wl.N  # the dense path: dQ-only main kernel, key-stationary dK/dV kernel
    if kernel == "sparse_fwd":
        return "tensor", 4.0 * BH * wl.N * wl.k * wl.d / launches_per_step, "flop"
    if kernel == "bwd_main":
        return "tensor", (6.0 if dense else 10.0) * BH * wl.N * wl.k * wl.d / launches_per_step, "flop"
    if kernel == "dense_dkdv":
        return "tensor", 8.0 * BH * wl.N * wl.N * wl.d / launches_per_step, "flop"
    if kernel == "dense_delta":
        return "hbm", (2.0 * BH * wl.N * wl.d * 2 + 4.0 * BH * wl.N) / launches_per_step, "byte"
    if kernel == "estimate_topk":
        return "hbm", (2.0 * BH * wl.N * wl.r * 2 + 4.0 * BH * wl.NB * wl.k) / launches_per_step, "byte"
    if kernel == "bwd_reduce":
        return "hbm", (pairs * (2 * wl.d * 2 + 4) + 2.0 * BH * wl.N * wl.d * 2) / launches_per_step, "byte"
    return None, None, None


def kernel_roofline(name, launches, total_ms, steps, wl):
    hbm, bf16, src = measured_peaks()
    bound, amount, unit = algorithmic(name, wl, launches / steps)
    out = {"kernel": name, "launches": launches, "avg_ms": total_ms / launches}
    if bound is None:
        out.update({"bound": None, "achieved": None, "peak": None, "unit": None, "frac": None})
        return out
    avg_s = total_ms / launches / 1e3
    if bound == "tensor":
        achieved = amount / avg_s / 1e12
        out.update({"bound": "tensor", "achieved": achieved, "peak": bf16, "unit": "TFLOP/s",
                    "frac": achieved / bf16, "peak_source": f"bf16_tflops burst, of {src}"})
    else:
        achieved = amount / avg_s / 1e9
        out.update({"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                    "peak_source": f"hbm_gbs, of {src}"})
    out["algorithmic_per_launch"] = amount
    return out


def roofline(prof, steps, wl):
    kern = {k: v for k, v in prof.items() if k != "dropped"}
    name, (launches, total_ms) = max(kern.items(), key=lambda kv: kv[1][1])
    out = kernel_roofline(name, launches, total_ms, steps, wl)
    out["share_of_kernel_time"] = total_ms / sum(v[1] for v in kern.values())
    traffic = None
    if os.path.exists(TRAFFIC_FILE):
        t = json.load(open(TRAFFIC_FILE)).get(name)
        if t and t.get("source_hash") == kernel_source_hash(name) and t.get("workload") == wl.name:
            # DRAM bytes per selected (block, key) pair of one captured launch, times this launch's pairs
            traffic = t["bytes_per_pair"] * wl.B * wl.H * wl.NB * wl.k / (launches / steps)
            out["traffic_source"] = t["how"]
    out["traffic"] = traffic
    if name == "bwd_main":
        # the same launches seen from HBM: every pair writes its bf16 partial row (4 d bytes) and list
        # entry, and gathers its K and V rows (4 d bytes, from L2 or HBM)
        pairs = wl.B * wl.H * wl.NB * wl.k / (launches / steps)
        hbm = measured_peaks()[0]
        w = pairs * (4 * wl.d + 4) / (out["avg_ms"] / 1e3) / 1e9
        out["hbm_view"] = {"partial_row_write_gbs": w, "frac_of_hbm": w / hbm,
                           "gather_gbs": pairs * 4 * wl.d / (out["avg_ms"] / 1e3) / 1e9}
    return out


# ---------------------------------------------------------------- side measurements

def adaln_measurements(dev, timed):
    """Fused AdaLN on its two workloads: forward and backward times (L2 flushed before each call),
    algorithmic bytes, achieved GB/s and the fraction of the measured HBM copy bandwidth."""
    import torch
    from dynamic_sparse_attention_estimate_gb300 import dsv_adaln_bwd, dsv_adaln_bwd_workspace, dsv_adaln_fwd
    from dynamic_sparse_attention_estimate_gb300.binding import dsv_profile_enable, dsv_profile_read
    from dynamic_sparse_attention_estimate_gb300.inputs import ADALN_WORKLOADS, make_adaln_inputs
    hbm = measured_peaks()[0]
    out = {}
    for name, (B, N, D) in sorted(ADALN_WORKLOADS.items()):
        g = {k: v.to(dev) for k, v in make_adaln_inputs(B, N, D).items()}
        y = torch.empty_like(g["x"])
        res = (torch.empty_like(g["x"]), torch.empty((B, D), dtype=torch.float32, device=dev),
               torch.empty((B, D), dtype=torch.float32, device=dev))
        ws = torch.empty(max(1, dsv_adaln_bwd_workspace(B, N, D)), dtype=torch.uint8, device=dev)
        fwd = lambda: dsv_adaln_fwd(g["x"], g["scale"], g["shift"], y=y)
        bwd = lambda: dsv_adaln_bwd(g["x"], g["scale"], g["dy"], out=res, workspace=ws)
        for _ in range(3):
            fwd()
            bwd()
        t_f, t_b = timed(fwd, 20), timed(bwd, 20)
        dsv_profile_enable(True)
        timed(fwd, 20)
        timed(bwd, 20)
        kernels = {k: v[1] / v[0] for k, v in dsv_profile_read().items() if k.startswith("adaln")}
        dsv_profile_enable(False)
        act = B * N * D * 2
        b_f = 2 * act + 2 * B * D * 2                  # x in, y out, scale and shift in
        b_b = 3 * act + B * D * 2 + 2 * B * D * 4      # x, dy in, dx out, scale in, d_scale and d_shift out
        out[name] = {"B": B, "N": N, "D": D, "fwd_ms": t_f, "bwd_ms": t_b, "fwd_bytes": b_f, "bwd_bytes": b_b,
                     "fwd_gbs": b_f / (t_f / 1e3) / 1e9, "bwd_gbs": b_b / (t_b / 1e3) / 1e9,
                     "fwd_frac_of_measured_hbm": b_f / (t_f / 1e3) / 1e9 / hbm,
                     "bwd_frac_of_measured_hbm": b_b / (t_b / 1e3) / 1e9 / hbm,
                     "kernel_ms": kernels, "workspace_bytes": ws.numel()}
        del g, y, res, ws
    return out


def dense_comparator(g, wl, flush_l2, ms_per_step):
    """PyTorch SDPA forward + backward (a library timing comparator, not this library) on the same
    per-head shape, every backend that runs here, one head, scaled to the step's heads; each
    backend's fastest call is kept and the speedup is quoted against the fastest backend."""
    import torch
    from torch.nn.attention import SDPBackend, sdpa_kernel
    heads = 1 if wl.N > 65536 else heads_per_call(wl)
    scale_to = wl.H / heads
    qf, kf, vf = [g[n][:, :heads].detach().clone().requires_grad_(True) for n in ("q", "k", "v")]
    do = g["do"][:, :heads].contiguous()
    dense_flop = 14.0 * wl.B * wl.H * wl.N * wl.N * wl.d
    reps = 3 if wl.N > 65536 else 5

    def fastest_of(fn, n):
        # the comparator's best call (its time varies between calls and runs): the speedup quoted
        # against it is the smallest one
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in ev:
            flush_l2()
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return min(a.elapsed_time(b) for a, b in ev)

    backends = {}
    for name, be in (("cudnn", SDPBackend.CUDNN_ATTENTION), ("flash", SDPBackend.FLASH_ATTENTION),
                     ("efficient", SDPBackend.EFFICIENT_ATTENTION)):
        try:
            def dense_step():
                with sdpa_kernel([be]):
                    out = torch.nn.functional.scaled_dot_product_attention(qf, kf, vf)
                    out.backward(do)
            dense_step()
            torch.cuda.synchronize()
            ms = fastest_of(dense_step, reps) * scale_to
            backends[name] = {"ms": ms, "tflops": dense_flop / (ms / 1e3) / 1e12}
        except Exception as exc:  # a backend that does not run on this GPU / shape
            backends[name] = {"error": str(exc).splitlines()[0][:160]}
        torch.cuda.synchronize()
    ok = {k: v for k, v in backends.items() if "ms" in v}
    out = {"impl": "torch SDPA (library), fwd+bwd", "heads_timed": heads,
           "scaled": f"x{scale_to:g} to the step's {wl.H} heads" if scale_to != 1 else None, "backends": backends}
    if ok:
        best = min(ok, key=lambda k: ok[k]["ms"])
        out.update({"fastest": best, "ms": ok[best]["ms"], "tflops": ok[best]["tflops"],
                    "speedup_of_sparse_step": ok[best]["ms"] / ms_per_step})
    del qf, kf, vf, do
    return out


def adaptive_measurement(dev, timed):
    """The mass-based selection (per block the keys carrying 90 % of the estimated mass, tau = 1/64)
    on the short clip: selection, then forward + backward over the CSR key lists."""
    import torch
    from dynamic_sparse_attention_estimate_gb300 import (dsv_estimate_mass_k, dsv_estimate_topk_csr,
                                                          dsv_sparse_attn_bwd_csr, dsv_sparse_attn_fwd_csr)
    from dynamic_sparse_attention_estimate_gb300.inputs import WORKLOADS, make_inputs_on_device
    wl = WORKLOADS["short"]
    g = make_inputs_on_device(wl, dev)
    o = torch.empty_like(g["q"])
    lse = torch.empty((wl.B, wl.H, wl.N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(o), torch.empty_like(o), torch.empty_like(o)
    k_row, rowptr, order = dsv_estimate_mass_k(g["q_lr"], g["k_lr"], 1.0 / 64, 0.9)
    cols = dsv_estimate_topk_csr(g["q_lr"], g["k_lr"], k_row, rowptr)
    pairs = cols.numel()
    ws_a = torch.empty(dsv_sparse_attn_bwd_csr_workspace_bytes(wl, pairs), dtype=torch.uint8, device=dev)
    t_sel = timed(lambda: (dsv_estimate_mass_k(g["q_lr"], g["k_lr"], 1.0 / 64, 0.9, out=(k_row, rowptr, order)),
                           dsv_estimate_topk_csr(g["q_lr"], g["k_lr"], k_row, rowptr, cols=cols)), 5)
    t_af = timed(lambda: dsv_sparse_attn_fwd_csr(g["q"], g["k"], g["v"], rowptr, cols, out=(o, lse), order=order), 5)
    t_ab = timed(lambda: dsv_sparse_attn_bwd_csr(g["do"], g["q"], g["k"], g["v"], o, lse, rowptr, cols,
                                                 workspace=ws_a, out=(dq, dk, dv), order=order), 5)
    fl_a = 14.0 * 64 * pairs * wl.d
    kr = k_row.float()
    return {"workload": "short clip (12 heads, N=16384, d=64)", "tau": 1.0 / 64, "mass": 0.9,
            "mean_k": float(kr.mean()), "min_k": int(k_row.min()), "max_k": int(k_row.max()),
            "density": pairs / (wl.B * wl.H * wl.NB * wl.N), "selection_ms": t_sel, "fwd_ms": t_af, "bwd_ms": t_ab,
            "attn_tflops": fl_a / ((t_af + t_ab) / 1e3) / 1e12,
            "step_tflops": fl_a / ((t_sel + t_af + t_ab) / 1e3) / 1e12}


# ---------------------------------------------------------------- the DSV arm

class LayerStep:
    """One step over every head of the layer, head group by head group: estimate -> forward ->
    backward.  When a group's backward fits one wave of the workspace, its first part (the key-major
    rank structure of idx) runs on a second stream beside the forward."""

    def __init__(self, wl, dev, ws_cap):
        import torch
        from dynamic_sparse_attention_estimate_gb300.binding import dsv_sparse_attn_bwd_workspace, make_dims
        self.wl, self.dev = wl, dev
        self.hpc = heads_per_call(wl)
        self.groups = [(h0, min(self.hpc, wl.H - h0)) for h0 in range(0, wl.H, self.hpc)]
        self.idx = torch.empty((wl.B, self.hpc, wl.NB, wl.k), dtype=torch.int32, device=dev)
        dims = make_dims(wl.B, self.hpc, wl.N, wl.d, wl.r, wl.k)
        one_wave = dsv_sparse_attn_bwd_csr_workspace_bytes(wl, wl.B * self.hpc * wl.NB * wl.k, self.hpc)
        ws_bytes = one_wave if one_wave <= ws_cap else max(dsv_sparse_attn_bwd_workspace(dims), int(ws_cap))
        self.split = ws_bytes >= one_wave
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        self.side = torch.cuda.Stream()
        self.have_idx, self.prepared = torch.cuda.Event(), torch.cuda.Event()

    def group(self, x, out, h0, nh, idx=None):
        """Estimate, forward and backward of heads [h0, h0 + nh) of the tensors in x, writing the
        matching heads of out (o, lse, dq, dk, dv), on the current stream."""
        import torch
        from dynamic_sparse_attention_estimate_gb300 import (dsv_estimate_topk, dsv_sparse_attn_bwd,
                                                             dsv_sparse_attn_bwd_prepare, dsv_sparse_attn_bwd_prepared,
                                                             dsv_sparse_attn_fwd)
        wl = self.wl
        sl = lambda t: t[:, h0:h0 + nh]
        idx = self.idx[:, :nh] if idx is None else idx
        q, k, v, do = sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["do"])
        o, lse, dq, dk, dv = (sl(out[n]) for n in ("o", "lse", "dq", "dk", "dv"))
        dsv_estimate_topk(sl(x["q_lr"]), sl(x["k_lr"]), wl.k, idx=idx)
        if self.split:
            cur = torch.cuda.current_stream()
            self.have_idx.record(cur)
            dsv_sparse_attn_fwd(q, k, v, idx, out=(o, lse))
            with torch.cuda.stream(self.side):
                self.side.wait_event(self.have_idx)
                dsv_sparse_attn_bwd_prepare(idx, wl.d, self.ws)
                self.prepared.record(self.side)
            cur.wait_event(self.prepared)
            dsv_sparse_attn_bwd_prepared(do, q, k, v, o, lse, idx, self.ws, out=(dq, dk, dv))
        else:
            dsv_sparse_attn_fwd(q, k, v, idx, out=(o, lse))
            dsv_sparse_attn_bwd(do, q, k, v, o, lse, idx, workspace=self.ws, out=(dq, dk, dv))

    def __call__(self, x, out):
        for h0, nh in self.groups:
            self.group(x, out, h0, nh)


def check_status(where):
    from dynamic_sparse_attention_estimate_gb300.binding import dsv_last_device_status
    st = dsv_last_device_status()
    if st != 0:
        raise RuntimeError(f"device status word set during {where} (status {st}): the run is not valid")


def dsv_arm(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from dynamic_sparse_attention_estimate_gb300 import (dsv_estimate_topk, dsv_sparse_attn_bwd,
                                                         dsv_sparse_attn_fwd, load_library)
    from dynamic_sparse_attention_estimate_gb300.binding import (dsv_profile_enable, dsv_profile_read,
                                                                 dsv_sparse_attn_bwd_workspace, make_dims)
    from dynamic_sparse_attention_estimate_gb300.inputs import make_inputs_on_device
    load_library()

    wl = workload(args)
    BH = wl.B * wl.H
    names = ("q", "k", "v", "do", "q_lr", "k_lr")
    g = make_inputs_on_device(wl, dev)
    outs = {"o": torch.empty_like(g["q"]), "lse": torch.empty((wl.B, wl.H, wl.N), dtype=torch.float32, device=dev),
            "dq": torch.empty_like(g["q"]), "dk": torch.empty_like(g["q"]), "dv": torch.empty_like(g["q"])}
    step = LayerStep(wl, dev, args.ws_gib * GIB)
    # L2 flush between timed calls: write a 512 MiB buffer (4x the 129 MB L2), then read another
    # one, so that the lines left in L2 are clean and the next timed kernel does not pay for
    # writing the flush's dirty lines back to HBM
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_rd = torch.zeros(128 << 20, dtype=torch.float32, device=dev)

    def flush_l2():
        flush.zero_()
        flush_rd.sum()

    if args.profile_once:
        step.group(g, outs, 0, step.groups[0][1])
        torch.cuda.synchronize()
        check_status("the profiled group")
        print(json.dumps({"profile_once": config_of(wl)["workload"], "heads": step.groups[0][1],
                          "workspace_gib": step.ws.numel() / GIB}), flush=True)
        return 0

    for _ in range(args.warmup):
        step(g, outs)
    torch.cuda.synchronize()
    check_status("warm-up")

    # ---- timed region (device-resident inputs)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall0 = time.time()
        dsv_profile_enable(True)
        for i in range(args.steps):
            flush_l2()
            starts[i].record()
            step(g, outs)
            ends[i].record()
        torch.cuda.synchronize()
        t_wall1 = time.time()
        prof = dsv_profile_read()
        dsv_profile_enable(False)
    clocks = clk.summary(t_wall0, t_wall1)
    check_status("the timed steps")
    total_ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends))
    if world > 1:
        dist.barrier()
    total_ms = max_over_ranks(total_ms, dev, world)
    fl = flops_per_step(wl)
    value = job_tflops(world, args.steps, fl, total_ms)
    ms_per_step = total_ms / args.steps
    heavy = ms_per_step > 300.0

    def timed(fn, n):
        """Median device time of fn over n calls, each after an L2 flush.  All n calls are
        enqueued before one synchronisation, so the host's launch latency stays outside the
        events (the flush ahead of each call gives the host time to enqueue)."""
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in ev:
            flush_l2()
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ev)

    # ---- stage breakdown: each stage over every head group, timed alone (same inputs)
    n_stage = 2 if heavy else max(3, min(20, args.steps))
    sl = lambda t, h0, nh: t[:, h0:h0 + nh]
    idx_all = [step.idx[:, :nh] for _, nh in step.groups]

    def est_all():
        for (h0, nh), idx in zip(step.groups, idx_all):
            dsv_estimate_topk(sl(g["q_lr"], h0, nh), sl(g["k_lr"], h0, nh), wl.k, idx=idx)

    def fwd_all():
        for (h0, nh), idx in zip(step.groups, idx_all):
            dsv_sparse_attn_fwd(sl(g["q"], h0, nh), sl(g["k"], h0, nh), sl(g["v"], h0, nh), idx,
                                out=(sl(outs["o"], h0, nh), sl(outs["lse"], h0, nh)))

    def bwd_all():
        for (h0, nh), idx in zip(step.groups, idx_all):
            dsv_sparse_attn_bwd(*(sl(g[n], h0, nh) for n in ("do", "q", "k", "v")), sl(outs["o"], h0, nh),
                                sl(outs["lse"], h0, nh), idx, workspace=step.ws,
                                out=tuple(sl(outs[n], h0, nh) for n in ("dq", "dk", "dv")))

    if len(step.groups) == 1:
        t_est, t_fwd, t_bwd = timed(est_all, n_stage), timed(fwd_all, n_stage), timed(bwd_all, n_stage)
    else:   # the selection of a group is overwritten by the next: time each group's stages in turn
        t_est = t_fwd = t_bwd = 0.0
        for gi in range(len(step.groups)):
            h0, nh = step.groups[gi]
            idx = idx_all[gi]
            t_est += timed(lambda: dsv_estimate_topk(sl(g["q_lr"], h0, nh), sl(g["k_lr"], h0, nh), wl.k, idx=idx),
                           n_stage)
            t_fwd += timed(lambda: dsv_sparse_attn_fwd(sl(g["q"], h0, nh), sl(g["k"], h0, nh), sl(g["v"], h0, nh),
                                                       idx, out=(sl(outs["o"], h0, nh), sl(outs["lse"], h0, nh))),
                           n_stage)
            t_bwd += timed(lambda: dsv_sparse_attn_bwd(*(sl(g[n], h0, nh) for n in ("do", "q", "k", "v")),
                                                       sl(outs["o"], h0, nh), sl(outs["lse"], h0, nh), idx,
                                                       workspace=step.ws,
                                                       out=tuple(sl(outs[n], h0, nh) for n in ("dq", "dk", "dv"))),
                           n_stage)
    check_status("the stage timings")

    # ---- e2e through the public API with host buffers: every head group's inputs are copied
    # host->device from pinned memory and its outputs (O, LSE, dQ, dK, dV) back, inside the timed
    # region.  Measured two ways: serial (copy in, compute, copy out, synchronise, group by group)
    # and pipelined (three streams, device buffers for two groups: group i+1's inputs go in and
    # group i-1's outputs come back while group i computes), which is what a training loop that
    # prefetches its batches sees.
    e2e = None
    if not args.no_e2e:
        pinned = {n: torch.empty(g[n].shape, dtype=g[n].dtype, pin_memory=True) for n in names}
        for n in names:
            pinned[n].copy_(g[n])
        back = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in outs.items()}
        h2d = sum(t.numel() * t.element_size() for t in pinned.values())
        d2h = sum(t.numel() * t.element_size() for t in back.values())
        n_e2e = 2 if heavy else max(3, min(args.steps, 50))
        hpc = step.hpc
        slots = []
        for _ in range(2):
            gi = {n: torch.empty((wl.B, hpc) + tuple(g[n].shape[2:]), dtype=g[n].dtype, device=dev) for n in names}
            go = {n: torch.empty((wl.B, hpc) + tuple(t.shape[2:]), dtype=t.dtype, device=dev)
                  for n, t in outs.items()}
            slots.append((gi, go, torch.empty_like(step.idx)))
        units = [(s, h0, nh) for s in range(n_e2e) for (h0, nh) in step.groups]

        def copy_in(gi, h0, nh):
            for n in names:
                gi[n][:, :nh].copy_(sl(pinned[n], h0, nh), non_blocking=True)

        def copy_out(go, h0, nh):
            for n in outs:
                sl(back[n], h0, nh).copy_(go[n][:, :nh], non_blocking=True)

        def compute(gi, go, idx_s, nh):
            step.group(gi, go, 0, nh, idx=idx_s[:, :nh])

        def serial(n_units):
            for i in range(n_units):
                _, h0, nh = units[i % len(units)]
                gi, go, idx_s = slots[0]
                copy_in(gi, h0, nh)
                compute(gi, go, idx_s, nh)
                copy_out(go, h0, nh)
                torch.cuda.synchronize()

        serial(len(step.groups))   # untimed
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        serial(len(units))
        b.record()
        torch.cuda.synchronize()
        serial_ms = max_over_ranks(a.elapsed_time(b), dev, world) / n_e2e

        s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        in_done = [torch.cuda.Event() for _ in range(2)]
        cmp_done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]

        def pipelined(n_units, t0=None, t1=None):
            for i in range(n_units):
                _, h0, nh = units[i % len(units)]
                si = i % 2
                gi, go, idx_s = slots[si]
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(cmp_done[si])      # unit i-2 has consumed this slot's inputs
                    if i == 0 and t0 is not None:
                        t0.record(s_in)
                    copy_in(gi, h0, nh)
                    in_done[si].record(s_in)
                with torch.cuda.stream(s_cmp):
                    s_cmp.wait_event(in_done[si])
                    if i >= 2:
                        s_cmp.wait_event(out_done[si])     # unit i-2's outputs have left this slot
                    compute(gi, go, idx_s, nh)
                    cmp_done[si].record(s_cmp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(cmp_done[si])
                    copy_out(go, h0, nh)
                    out_done[si].record(s_out)
            if t1 is not None:
                with torch.cuda.stream(s_out):
                    t1.record(s_out)
            torch.cuda.synchronize()

        # the copies alone (every unit's H2D then D2H, no compute), to show what the pipeline hides
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        c0.record()
        for i, (_, h0, nh) in enumerate(units):
            gi, go, _ = slots[i % 2]
            copy_in(gi, h0, nh)
            copy_out(go, h0, nh)
        c1.record()
        torch.cuda.synchronize()
        copy_ms = max_over_ranks(c0.elapsed_time(c1), dev, world) / n_e2e

        pipelined(min(2, len(units)))               # untimed
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        # the start event waits for nothing queued before it: every stream is idle here
        pipelined(len(units), t0, t1)
        pipe_ms = max_over_ranks(t0.elapsed_time(t1), dev, world) / n_e2e
        check_status("the end-to-end steps")
        e2e = {"value": job_tflops(world, n_e2e, fl, pipe_ms * n_e2e), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": pipe_ms, "steps": n_e2e,
               "pipelined": "3 streams; device buffers for two head groups; group i+1's H2D and group i-1's D2H "
                            "overlap group i's estimate, forward and backward",
               "copies_alone_ms_per_step": copy_ms,
               "serial": {"value": job_tflops(world, n_e2e, fl, serial_ms * n_e2e), "ms_per_step": serial_ms}}
        del pinned, back, slots

    side = not args.no_side
    dense = None
    if side and not args.no_dense:
        try:
            dense = dense_comparator(g, wl, flush_l2, ms_per_step)
        except Exception as exc:  # a comparator only
            dense = {"error": str(exc)[:200]}

    # ---- this library at density 100 % (k = N: every key selected) on the same shape: its dense path
    # (key-stationary dK / dV, no idx, no partial rows), one head for the long shapes, scaled
    own_dense = None
    if side and not args.no_dense:
        try:
            heads = 1 if wl.N > 65536 else step.hpc
            sl1 = lambda t: t[:, :heads]
            ws_d = torch.empty(max(1, dsv_sparse_attn_bwd_workspace(make_dims(wl.B, heads, wl.N, wl.d, wl.r, wl.N))),
                               dtype=torch.uint8, device=dev)

            def own_dense_step():
                dsv_sparse_attn_fwd(sl1(g["q"]), sl1(g["k"]), sl1(g["v"]), None,
                                    out=(sl1(outs["o"]), sl1(outs["lse"])))
                dsv_sparse_attn_bwd(*(sl1(g[n]) for n in ("do", "q", "k", "v")), sl1(outs["o"]), sl1(outs["lse"]),
                                    None, workspace=ws_d, out=tuple(sl1(outs[n]) for n in ("dq", "dk", "dv")))
            own_dense_step()
            t_od = timed(own_dense_step, 2 if wl.N > 65536 else 5) * (wl.H / heads)
            dense_flop = 14.0 * BH * wl.N * wl.N * wl.d
            own_dense = {"ms": t_od, "tflops": dense_flop / (t_od / 1e3) / 1e12, "heads_timed": heads,
                         "impl": "this library at k = N: forward without idx, dense dK/dV kernel + dQ-only main kernel",
                         "scaled": f"x{wl.H / heads:g} to the step's {wl.H} heads" if heads != wl.H else None}
            if dense and "ms" in dense:
                own_dense["vs_fastest_sdpa"] = dense["ms"] / t_od
            del ws_d
        except Exception as exc:  # a comparator only
            own_dense = {"error": str(exc)[:200]}
        check_status("the dense comparison")

    adaptive = None
    if side and not args.no_adaptive:
        try:
            adaptive = adaptive_measurement(dev, timed)
        except Exception as exc:  # a side measurement only
            adaptive = {"error": str(exc)[:200]}

    # ---- fused AdaLN (LayerNorm + modulation) forward and backward, HBM-bound: bytes moved per
    # call (x, dy read; y, dx written; modulation vectors and gradients) over the measured time
    adaln = None
    if side and not args.no_adaln:
        try:
            adaln = adaln_measurements(dev, timed)
        except Exception as exc:  # a side measurement only
            adaln = {"error": str(exc)[:200]}
    check_status("the side measurements")

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        fl_s, dt, nb = oracle_sample(wl, 12.0)
        cpu = {"value": fl_s / dt / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{nb} of {BH * wl.NB} query blocks (head 0): estimate + forward + backward, numpy fp64, "
                         f"{dt:.1f} s"}

    rl = roofline(prof, args.steps, wl)
    launches = sum(v[0] for k, v in prof.items() if k != "dropped")
    hbm, bf16, src = measured_peaks()
    kernels = {k: kernel_roofline(k, v[0], v[1], args.steps, wl) for k, v in prof.items() if k != "dropped"}
    for k, v in kernels.items():
        v["ms_per_step"] = prof[k][1] / args.steps
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": f"synthetic (seeded; drawn on the device by torch's generator with the {wl.name} workload's "
                f"distributions, shapes and block-major order)",
        "config": config_of(wl),
        "step": ("per group of %d heads: estimate; forward; %s" % (
            step.hpc, "the backward's rank structure of idx on a second stream beside the forward, then the rest "
                      "of the backward" if step.split else "the backward (waves of query blocks through a %.0f GiB "
                                                            "workspace)" % (step.ws.numel() / GIB))),
        "tokens_per_s": world * wl.B * wl.N * args.steps / (total_ms / 1e3),
        "pct_of_bf16_peak": 100.0 * value / world / bf16,
        "stages_ms": {"estimate_topk": t_est, "sparse_fwd": t_fwd, "sparse_bwd": t_bwd},
        "attn_only_tflops": 14.0 * BH * wl.N * wl.k * wl.d / ((t_fwd + t_bwd) / 1e3) / 1e12,
        "tokens_per_s_attn_only": wl.B * wl.N / ((t_fwd + t_bwd) / 1e3),
        "kernels": kernels,
        "kernel_ms_note": "per-kernel event times inside the timed steps; kernels on the second stream (the "
                          "backward's set_bits, colpre, scan beside the forward) include waiting for SMs",
        "estimate": {"ms": t_est, "score_elements_per_s": BH * wl.NB * wl.N / (t_est / 1e3),
                     "mma_tflops": 2.0 * wl.r * BH * wl.NB * wl.N / (t_est / 1e3) / 1e12},
        "roofline": rl, "gpu_launches": launches, "clocks": clocks, "e2e": e2e, "dense_comparator": dense,
        "own_dense_path": own_dense, "adaptive_selection": adaptive, "adaln": adaln,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return reference_arm(args)
    return dsv_arm(args)


if __name__ == "__main__":
    sys.exit(main())
