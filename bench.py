#!/usr/bin/env python3
"""Benchmark of the fused LayerNorm / RMSNorm library on one GB300.

Headline step (one pass of the hot path over one batch): LayerNorm forward
with fused FP8 delayed-scaling output, then LayerNorm backward (dx, dgamma,
dbeta), zero-centered gamma, x and dz bf16 [8192 x 4096] (synthetic, seeded,
rn_inputs workload "ln_delayed").  Metric: effective HBM GB/s, i.e.
algorithmic bytes (every input read once, every output written once) per
second of kernel time, with L2 flushed before each forward and each backward.

Also reported (key "workloads"): the other workloads at full size, each as
GB/s, rows/s and the fraction of the HBM peak.

Usage:  python bench.py [--steps K] [--warmup W] [--impl rn|reference]
Multi-GPU (torchrun): every rank runs the same workload independently
(replicas; the path has no exchange step on one node's data here).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
PROFILE_DIR = os.path.join(ROOT, "profiles")
METRIC = "norm fwd/bwd effective HBM GB/s (+rows/s) and % of GB300 8 TB/s peak, 1 GPU"


# ------------------------------------------------------------------ helpers
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            flat = {}

            def walk(o, pre=""):
                if isinstance(o, dict):
                    for k, v in o.items():
                        walk(v, f"{pre}{k}.")
                else:
                    flat[pre[:-1]] = o
            walk(d)
            for k, v in flat.items():
                if "hbm" in k.lower() and isinstance(v, (int, float)) and v > 100:
                    return float(v), "measured", k
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback", None


def algorithmic_bytes(kind, N, H, esz, ln, extra=None):
    """Bytes every kernel must move at least once (inputs read, outputs written)."""
    E = N * H
    vec = H * 4 * (2 if ln else 1)          # gamma (+ beta) fp32
    stats = N * 4 * (2 if ln else 1)        # mu (+) rsigma fp32
    if kind == "fwd_none":
        return E * esz + E * esz + vec + stats
    if kind == "fwd_fp8":                    # x in, codes out
        return E * esz + E * 1 + vec + stats
    if kind == "fwd_fp8_current":            # x read twice (amax pass, quantize pass)
        return 2 * E * esz + E * 1 + vec + 2 * stats
    if kind == "fwd_nvfp4":                  # x read twice; E2M1 codes (half a byte) and scales out
        return 2 * E * esz + E // 2 + E // 16 + vec + 2 * stats
    if kind == "fwd_mxfp8_row":              # x in, rowwise codes and scales out
        return E * esz + E + E // 32 + vec + stats
    if kind == "fwd_mxfp8":                  # x in, row + col codes and scales out
        return E * esz + 2 * E + 2 * (E // 32) + vec + stats
    if kind == "bwd":                        # dz, x in, dx out, dgamma (+dbeta) out
        return 3 * E * esz + stats + H * 4 + vec
    if kind == "fwd_add_fp8":                # x, residual in; h and codes out
        return 3 * E * esz + E * 1 + vec + stats
    if kind == "fwd_add_mxfp8":              # x, residual in; h, row + col codes and scales out
        return 3 * E * esz + 2 * E + 2 * (E // 32) + vec + stats
    # scaled SwiGLU, E = N x H outputs from N x 2H inputs, row scales fp32
    if kind == "act_fwd_none":               # x in (2E), y out
        return 2 * E * esz + E * esz + 4 * N
    if kind == "act_fwd_fp8_current":        # x read twice, E4M3 codes out
        return 2 * (2 * E * esz + 4 * N) + E
    if kind == "act_fwd_mxfp8":              # x in, rowwise codes + E8M0 scales out
        return 2 * E * esz + E + E // 32 + 4 * N
    if kind == "act_bwd":                    # dy, x in; dx out (2E); scales in, dscales out
        return E * esz + 2 * E * esz + 2 * E * esz + 8 * N
    if kind == "history":                    # history read + written (H entries), 3 scalars
        return 2 * H * 4 + 12
    raise ValueError(kind)


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "mxfp8_quantization_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def profile_traffic(name, files):
    """dram bytes per launch from a committed ncu summary, if the kernel
    source still matches the hash recorded with it; else None."""
    path = os.path.join(PROFILE_DIR, name)
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    hsh = re.search(r"source_hash:\s*([0-9a-f]+)", txt)
    if not m or not hsh or hsh.group(1) != kernel_source_hash(files):
        return None
    return float(m.group(1))


# Roofline entries for the largest shape of every forward mode and of the
# backward: (entry, workload result, kernels of the call, ncu summaries in
# profiles/ whose traffic adds up to the call's, kernel source files).
FWD_SRC = ["rn_fwd.cu", "rn_device.cuh"]
ROOFLINES = [
    ("rms_fwd_fp8_current_16384x8192", "rms_16384x8192_fwd_fp8_current",
     "rn_rmsnorm_fwd FP8_CURRENT: rn_fwd_init_kernel + rn_fwd_kernel (amax pass) + rn_fwd_kernel (quantize pass)",
     ["rn_fwd_rms_fp8_current_pass1_bf16_16384x8192.md", "rn_fwd_rms_fp8_current_pass2_bf16_16384x8192.md"],
     FWD_SRC),
    ("ln_fwd_mxfp8_65536x2048", "ln_65536x2048_fwd_mxfp8",
     "rn_layernorm_fwd MXFP8 rowwise + columnwise: rn_mx_box_kernel",
     ["rn_mx_ln_bf16_65536x2048.md"], ["rn_mx.cu", "rn_device.cuh"]),
    ("rms_fwd_mxfp8_65536x2048", "rms_65536x2048_fwd_mxfp8",
     "rn_rmsnorm_fwd MXFP8 rowwise + columnwise: rn_mx_box_kernel",
     ["rn_mx_rms_bf16_65536x2048.md"], ["rn_mx.cu", "rn_device.cuh"]),
    ("ln_fwd_mxfp8_rowwise_65536x2048", "ln_65536x2048_fwd_mxfp8_rowwise_only",
     "rn_layernorm_fwd MXFP8 rowwise only: rn_fwd_kernel",
     ["rn_fwd_ln_mxfp8_row_bf16_65536x2048.md"], FWD_SRC),
    ("ln_fwd_none_65536x2048", "ln_65536x2048_fwd_none", "rn_layernorm_fwd NONE: rn_fwd_kernel",
     ["rn_fwd_ln_none_bf16_65536x2048.md"], FWD_SRC),
    ("rms_fwd_none_65536x2048", "rms_65536x2048_fwd_none", "rn_rmsnorm_fwd NONE: rn_fwd_kernel",
     ["rn_fwd_rms_none_bf16_65536x2048.md"], FWD_SRC),
    ("rms_fwd_none_16384x8192", "rms_16384x8192_fwd_none", "rn_rmsnorm_fwd NONE: rn_fwd_kernel",
     ["rn_fwd_rms_none_bf16_16384x8192.md"], FWD_SRC),
    ("ln_fwd_fp8_delayed_65536x2048", "ln_65536x2048_fwd_fp8_delayed",
     "rn_layernorm_fwd FP8_DELAYED: rn_fwd_init_kernel + rn_fwd_kernel",
     ["rn_fwd_ln_fp8_delayed_bf16_65536x2048.md"], FWD_SRC),
    ("rms_fwd_fp8_delayed_65536x2048", "rms_65536x2048_fwd_fp8_delayed",
     "rn_rmsnorm_fwd FP8_DELAYED: rn_fwd_init_kernel + rn_fwd_kernel",
     ["rn_fwd_rms_fp8_delayed_bf16_65536x2048.md"], FWD_SRC),
    ("rms_fwd_fp8_delayed_16384x8192", "rms_16384x8192_fwd_fp8_delayed",
     "rn_rmsnorm_fwd FP8_DELAYED: rn_fwd_init_kernel + rn_fwd_kernel",
     ["rn_fwd_rms_fp8_delayed_bf16_16384x8192.md"], FWD_SRC),
    ("ln_bwd_f32_131072x1024", "ln_131072x1024_f32_bwd_margin0",
     "rn_layernorm_bwd fp32: rn_bwd_fused_kernel + rn_colreduce_kernel",
     ["rn_bwd_fused_ln_f32_131072x1024.md"], ["rn_bwd.cu", "rn_device.cuh"]),
    ("rms_bwd_f32_131072x1024", "rms_131072x1024_f32_bwd_margin0",
     "rn_rmsnorm_bwd fp32: rn_bwd_fused_kernel + rn_colreduce_kernel",
     ["rn_bwd_fused_rms_f32_131072x1024.md"], ["rn_bwd.cu", "rn_device.cuh"]),
    ("ln_bwd_bf16_3000x5120", "ln_3000x5120_bf16_bwd_margin0",
     "rn_layernorm_bwd bf16: rn_bwd_kernel + rn_colreduce_kernel",
     ["rn_bwd_ln_bf16_3000x5120.md"], ["rn_bwd.cu", "rn_device.cuh"]),
]


def roofline_entry(kernel, ms, algo_bytes, peak, peak_kind, profiles, files):
    """achieved = algorithmic bytes / mean call time (CUDA events); traffic =
    the sum of the committed ncu summaries' DRAM bytes per launch, or None
    when one is missing or older than the kernel source."""
    gbs = algo_bytes / (ms * 1e-3) / 1e9
    tr = [profile_traffic(f, files) for f in profiles]
    return {"kernel": kernel, "bound": "hbm", "achieved": round(gbs, 1), "peak": peak,
            "peak_kind": peak_kind, "unit": "GB/s", "frac": round(gbs / peak, 4),
            "traffic": None if any(t is None for t in tr) else int(sum(tr)),
            "algorithmic_bytes": algo_bytes, "ms": round(ms, 5), "profiles": profiles}


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=5)
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 8]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() in ("active", "1"):
                    reasons.add(n)
        # samples are taken every 20 ms across warm-up and the timed loop;
        # the loop itself is short, so all samples under load are reported
        loaded = [s for s in sm if s > 0]
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(rows)}


def aggregate_ranks(ms_per_step, bytes_per_step, dist=None, device="cpu"):
    """Whole-job figures of a replicas run: the slowest rank's time per step
    (max over ranks) and the bytes of all ranks over it.  Returns
    (max_ms, GB/s).  Without a process group: this rank alone."""
    import torch
    world = 1
    if dist is not None and dist.is_available() and dist.is_initialized():
        world = dist.get_world_size()
        t = torch.tensor([float(ms_per_step)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_per_step = float(t.item())
    return ms_per_step, world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


# ---------------------------------------------------------------- our arm
class Prepared:
    """Device buffers and ctypes argument lists for repeated C-ABI calls."""

    def __init__(self, rn, torch, w, ln=True):
        self.rn, self.torch, self.w, self.ln = rn, torch, w, ln
        dev = "cuda"
        bf16 = w.dtype == "bf16"
        tdt = torch.bfloat16 if bf16 else torch.float32
        to = (lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)) if bf16 \
            else (lambda a: torch.from_numpy(a).to(dev))
        self.x = to(w.x)
        self.dz = to(w.dz) if w.dz is not None else None
        self.gamma = torch.from_numpy(w.gamma).to(dev)
        self.beta = torch.from_numpy(w.beta).to(dev) if (ln and w.beta is not None) else None
        N, H = w.N, w.H
        self.N, self.H, self.esz = N, H, (2 if bf16 else 4)
        self.mu = torch.empty(N, dtype=torch.float32, device=dev)
        self.rs = torch.empty(N, dtype=torch.float32, device=dev)
        self.dtype_code = 0 if bf16 else 1
        self.tdt = tdt

    def stream(self):
        return ctypes.c_void_p(self.torch.cuda.current_stream().cuda_stream)

    def fwd_args(self, mode, scale=None):
        rn, torch = self.rn, self.torch
        o = rn._Output()
        N, H = self.N, self.H
        keep = []
        if mode == "fp8_delayed":
            data = torch.empty((N, H), dtype=torch.uint8, device="cuda")
            self.scale_t = torch.tensor([scale], dtype=torch.float32, device="cuda")
            sinv = torch.empty(1, dtype=torch.float32, device="cuda")
            amax = torch.empty(1, dtype=torch.float32, device="cuda")
            o.data, o.scale, o.scale_inv, o.amax = (data.data_ptr(), self.scale_t.data_ptr(),
                                                    sinv.data_ptr(), amax.data_ptr())
            keep = [data, sinv, amax]
        elif mode == "fp8_current":
            data = torch.empty((N, H), dtype=torch.uint8, device="cuda")
            sc, sinv, amax = (torch.empty(1, dtype=torch.float32, device="cuda") for _ in range(3))
            o.data, o.scale_out, o.scale_inv, o.amax = (data.data_ptr(), sc.data_ptr(),
                                                        sinv.data_ptr(), amax.data_ptr())
            keep = [data, sc, sinv, amax]
        elif mode == "nvfp4":
            d = torch.empty((N, H // 2), dtype=torch.uint8, device="cuda")
            rsc = torch.empty((N, H // 16), dtype=torch.uint8, device="cuda")
            sc, sinv, amax = (torch.empty(1, dtype=torch.float32, device="cuda") for _ in range(3))
            o.data, o.row_scales, o.scale_out, o.scale_inv, o.amax = (
                d.data_ptr(), rsc.data_ptr(), sc.data_ptr(), sinv.data_ptr(), amax.data_ptr())
            keep = [d, rsc, sc, sinv, amax]
        elif mode == "mxfp8_row":
            d = torch.empty((N, H), dtype=torch.uint8, device="cuda")
            rsc = torch.empty((N, H // 32), dtype=torch.uint8, device="cuda")
            o.data, o.row_scales = d.data_ptr(), rsc.data_ptr()
            keep = [d, rsc]
        elif mode == "mxfp8":
            d = torch.empty((N, H), dtype=torch.uint8, device="cuda")
            rsc = torch.empty((N, H // 32), dtype=torch.uint8, device="cuda")
            cd = torch.empty((H, N), dtype=torch.uint8, device="cuda")
            csc = torch.empty((H, N // 32), dtype=torch.uint8, device="cuda")
            o.data, o.row_scales, o.col_data, o.col_scales = (d.data_ptr(), rsc.data_ptr(),
                                                              cd.data_ptr(), csc.data_ptr())
            keep = [d, rsc, cd, csc]
        else:
            data = torch.empty((N, H), dtype=self.tdt, device="cuda")
            o.data, o.out_dtype = data.data_ptr(), self.dtype_code
            keep = [data]
        self.fwd_keep = keep
        self.fwd_out = o
        mcode = rn.QUANT_MODES["mxfp8" if mode == "mxfp8_row" else mode]
        w = self.w
        vp = ctypes.c_void_p
        if self.ln:
            return ("rn_layernorm_fwd",
                    [vp(self.x.data_ptr()), self.dtype_code, vp(self.gamma.data_ptr()),
                     vp(self.beta.data_ptr()) if self.beta is not None else None, N, H,
                     ctypes.c_float(w.eps), int(w.zero_centered_gamma), 0, mcode,
                     ctypes.byref(o), vp(self.mu.data_ptr()), vp(self.rs.data_ptr())])
        return ("rn_rmsnorm_fwd",
                [vp(self.x.data_ptr()), self.dtype_code, vp(self.gamma.data_ptr()), N, H,
                 ctypes.c_float(w.eps), int(w.zero_centered_gamma), 0, mcode, ctypes.byref(o),
                 vp(self.rs.data_ptr())])

    def add_args(self, mode, scale=None):
        """rn_rmsnorm_add_fwd / rn_layernorm_add_fwd: h = x + residual
        (stored), then the norm of h with output `mode`."""
        torch, w = self.torch, self.w
        to = (lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to("cuda")) \
            if w.dtype == "bf16" else (lambda a: torch.from_numpy(a).to("cuda"))
        self.res = to(w.residual)
        self.h = torch.empty_like(self.x)
        fn, args = self.fwd_args(mode, scale)
        vp = ctypes.c_void_p
        if self.ln:
            # (x, dtype, gamma, beta, N, H, eps, zcg, margin, mode, out, mu, rs)
            return ("rn_layernorm_add_fwd",
                    [args[0], vp(self.res.data_ptr())] + args[1:11] + [vp(self.h.data_ptr())] + args[11:])
        # (x, dtype, gamma, N, H, eps, zcg, margin, mode, out, rs)
        return ("rn_rmsnorm_add_fwd",
                [args[0], vp(self.res.data_ptr())] + args[1:10] + [vp(self.h.data_ptr())] + args[10:])

    def bwd_args(self, sm_margin=0):
        rn, torch = self.rn, self.torch
        N, H = self.N, self.H
        need = rn.bwd_workspace_bytes(N, H, self.tdt, self.ln)
        self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
        self.wsn = ctypes.c_size_t(self.ws.numel())
        self.dx = torch.empty((N, H), dtype=self.tdt, device="cuda")
        self.dg = torch.empty(H, dtype=torch.float32, device="cuda")
        self.db = torch.empty(H, dtype=torch.float32, device="cuda")
        vp = ctypes.c_void_p
        w = self.w
        if self.ln:
            return ("rn_layernorm_bwd",
                    [vp(self.dz.data_ptr()), vp(self.x.data_ptr()), self.dtype_code,
                     vp(self.mu.data_ptr()), vp(self.rs.data_ptr()), vp(self.gamma.data_ptr()), N, H,
                     int(w.zero_centered_gamma), sm_margin, vp(self.dx.data_ptr()),
                     vp(self.dg.data_ptr()), vp(self.db.data_ptr()), vp(self.ws.data_ptr()),
                     ctypes.byref(self.wsn)])
        return ("rn_rmsnorm_bwd",
                [vp(self.dz.data_ptr()), vp(self.x.data_ptr()), self.dtype_code,
                 vp(self.rs.data_ptr()), vp(self.gamma.data_ptr()), N, H,
                 int(w.zero_centered_gamma), sm_margin, vp(self.dx.data_ptr()),
                 vp(self.dg.data_ptr()), vp(self.ws.data_ptr()), ctypes.byref(self.wsn)])


def call(lib, fa, stream):
    fn, args = fa
    st = getattr(lib, fn)(*args, stream)
    if st != 0:
        raise RuntimeError(f"{fn} failed with status {st}")


def time_calls(torch, lib, calls, steps, warmup, flush):
    """Time each call in `calls` (list of (name, fa)) per step with CUDA events
    on the launching stream; L2 is flushed before every call (untimed)."""
    s = torch.cuda.current_stream()
    stream = ctypes.c_void_p(s.cuda_stream)
    for _ in range(warmup):
        for _, fa in calls:
            flush()
            call(lib, fa, stream)
    torch.cuda.synchronize()
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in calls] for _ in range(steps)]
    for k in range(steps):
        for (name, fa), (a, b) in zip(calls, ev[k]):
            flush()
            a.record(s)
            call(lib, fa, stream)
            b.record(s)
    torch.cuda.synchronize()
    return {name: [ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(steps)]
            for i, (name, _) in enumerate(calls)}


def l2_writeback_ms(torch, lib, fa, flush, reps=10):
    """Estimate of the write-back a call leaves for later: at 8192 x 4096 part
    of the call's output is still dirty in L2 (129 MB) when its end event
    fires, and the next flush writes it to HBM outside the timed region.
    Returns the mean flush time right after the call minus right after
    another flush (ms, >= 0)."""
    s = torch.cuda.current_stream()
    stream = ctypes.c_void_p(s.cuda_stream)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed_flush():
        a.record(s)
        flush()
        b.record(s)
        torch.cuda.synchronize()
        return a.elapsed_time(b)
    after_call, after_flush = [], []
    for _ in range(reps):
        flush()
        call(lib, fa, stream)
        after_call.append(timed_flush())
        flush()
        after_flush.append(timed_flush())
    return max(0.0, statistics.mean(after_call) - statistics.mean(after_flush))


def run_rn(args):
    import torch
    import torch.distributed as dist

    import mxfp8_quantization_gb300 as rn
    import rn_inputs
    from mxfp8_quantization_gb300 import _build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if args.only is not None:
        _build.build()
        lib = rn._load()
        l2 = torch.cuda.get_device_properties(local).L2_cache_size
        fb = torch.empty(2 * l2, dtype=torch.uint8, device="cuda")
        rb = torch.ones(2 * l2 // 4, dtype=torch.float32, device="cuda")

        def flush_only():
            fb.fill_(1)
            rb.sum()
        res = run_other_workloads(torch, rn, lib, rn_inputs, flush_only, hbm_peak()[0], args.steps,
                                  args.warmup, only=args.only)
        print(json.dumps({"only": args.only, "workloads": res}))
        return
    if world > 1:
        dist.init_process_group("nccl")
    if rank == 0 or world == 1:
        _build.build()
    if world > 1:
        dist.barrier()
    lib = rn._load()

    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device="cuda")
    read_buf = torch.ones(2 * l2 // 4, dtype=torch.float32, device="cuda")

    def flush():
        # write 2x L2, then read another 2x L2: the write evicts everything,
        # the read evicts the dirty lines of the write, so the timed call
        # starts with an L2 holding only clean, unrelated lines
        flush_buf.fill_(1)
        read_buf.sum()

    peak, peak_kind, peak_key = hbm_peak()

    # ---------------------------------------------------- headline workload
    w = rn_inputs.make("ln_delayed")
    N, H = w.N, w.H
    P = Prepared(rn, torch, w, ln=True)
    fwd = P.fwd_args("fp8_delayed", scale=w.scale)
    bwd = P.bwd_args()
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    times = time_calls(torch, lib, [("fwd", fwd), ("bwd", bwd)], args.steps, args.warmup, flush)
    t_wall = time.time() - t_wall0
    clocks = sampler.stop()
    fwd_ms = statistics.mean(times["fwd"])
    bwd_ms = statistics.mean(times["bwd"])
    b_fwd = algorithmic_bytes("fwd_fp8", N, H, 2, True)
    b_bwd = algorithmic_bytes("bwd", N, H, 2, True)
    step_bytes = b_fwd + b_bwd
    ms_step, value = aggregate_ranks(fwd_ms + bwd_ms, step_bytes, dist if world > 1 else None, "cuda")
    if world > 1:
        t = torch.tensor([fwd_ms, bwd_ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        fwd_ms, bwd_ms = (float(v) for v in t.tolist())

    wb_fwd = l2_writeback_ms(torch, lib, fwd, flush)
    wb_bwd = l2_writeback_ms(torch, lib, bwd, flush)

    # ------------------------------------------------ end to end, host data
    e2e = None
    if rank == 0:
        e2e = run_e2e(torch, lib, P, fwd, bwd, w, max(3, min(args.steps, 20)), step_bytes)

    # ------------------------------------------------------ other workloads
    extra = {}
    if not args.quick and rank == 0:
        extra = run_other_workloads(torch, rn, lib, rn_inputs, flush, peak,
                                    max(3, min(args.steps, 20)), args.warmup)

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return
    cpu = cpu_baseline(w, step_bytes) if not args.no_cpu else None
    pk = f"{peak_kind}" + (f" ({peak_key})" if peak_key else "")
    rooflines = {
        "ln_fwd_fp8_delayed_8192x4096": roofline_entry(
            "rn_layernorm_fwd FP8_DELAYED: rn_fwd_init_kernel + rn_fwd_kernel", fwd_ms, b_fwd, peak, pk,
            ["rn_fwd_ln_fp8_delayed_bf16_8192x4096.md"], FWD_SRC),
        "ln_bwd_bf16_8192x4096": roofline_entry(
            "rn_layernorm_bwd bf16: rn_bwd_kernel + rn_colreduce_kernel", bwd_ms, b_bwd, peak, pk,
            ["rn_bwd_ln_bf16_8192x4096.md"], ["rn_bwd.cu", "rn_device.cuh"]),
    }
    for name, key, kernel, profs, files in ROOFLINES:
        if key in extra:
            r = extra[key]
            rooflines[name] = roofline_entry(kernel, r["ms"], r["algorithmic_bytes"], peak, pk, profs, files)
    bwd_gbs = b_bwd / (bwd_ms * 1e-3) / 1e9
    fwd_gbs = b_fwd / (fwd_ms * 1e-3) / 1e9
    traffic = profile_traffic("rn_bwd_ln_bf16_8192x4096.md", ["rn_bwd.cu", "rn_device.cuh"])
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded rn_inputs workload ln_delayed)",
        "config": {"workload": "LayerNorm fwd (fused FP8 E4M3 delayed scaling, zero-centered gamma) "
                               "+ bwd, x/dz bf16 [8192 x 4096]",
                   "rows": N, "hidden": H, "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "l2": "flushed (2x L2 write) before every fwd and bwd call, outside the timed events",
                   "rows_per_s": round(world * N / (ms_step * 1e-3), 1),
                   "fwd_ms": round(fwd_ms, 6), "bwd_ms": round(bwd_ms, 6),
                   "fwd_GBps": round(fwd_gbs, 1), "bwd_GBps": round(bwd_gbs, 1),
                   "algorithmic_bytes_per_step": step_bytes,
                   "pct_of_8TBps": round(100 * value / world / 8000.0, 2),
                   "wall_s_timed_loop": round(t_wall, 3),
                   "l2_writeback_ms_est": {"fwd": round(wb_fwd, 5), "bwd": round(wb_bwd, 5)},
                   "GBps_if_writeback_timed": round(world * step_bytes / ((ms_step + wb_fwd + wb_bwd) * 1e-3)
                                                    / 1e9, 1)},
        "roofline": {"kernel": "rn_layernorm_bwd call (rn_bwd_kernel + rn_colreduce_kernel)",
                     "bound": "hbm", "achieved": round(bwd_gbs, 1), "peak": peak,
                     "peak_kind": f"{peak_kind}" + (f" ({peak_key})" if peak_key else ""),
                     "unit": "GB/s", "frac": round(bwd_gbs / peak, 4),
                     "traffic": traffic, "algorithmic_bytes": b_bwd},
        "roofline_fwd": {"kernel": "rn_layernorm_fwd call (rn_fwd_kernel, FP8 delayed)",
                         "bound": "hbm", "achieved": round(fwd_gbs, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(fwd_gbs / peak, 4),
                         "traffic": profile_traffic("rn_fwd_ln_fp8_delayed_bf16_8192x4096.md",
                                                    ["rn_fwd.cu", "rn_device.cuh"]),
                         "algorithmic_bytes": b_fwd},
        "rooflines": rooflines,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 4 * args.steps,  # init + forward, backward + column reduction
        "clocks": clocks,
        "workloads": extra,
    }
    print(json.dumps(line))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_e2e(torch, lib, P, fwd, bwd, w, steps, step_bytes):
    """Same step through the C ABI with host data: every step copies its
    inputs in from pinned host memory and all of its results out, inside the
    timed region.  Steps are pipelined as a user would: the copy-out of step
    k runs on a second stream while step k + 1 copies its inputs in (the two
    directions of the host link overlap; copying x and dz in on two streams
    gained nothing: the copy-in is bound by the link); step k + 1's kernels
    wait for step k's copy-out, since they overwrite the same output
    buffers."""
    hx = torch.empty(P.x.shape, dtype=P.x.dtype, pin_memory=True)
    hx.copy_(P.x.cpu())
    hdz = torch.empty(P.dz.shape, dtype=P.dz.dtype, pin_memory=True)
    hdz.copy_(P.dz.cpu())
    hg = P.gamma.cpu().pin_memory()
    hb = P.beta.cpu().pin_memory()
    outs = [P.fwd_keep[0], P.mu, P.rs, P.fwd_keep[2], P.dx, P.dg, P.db]
    houts = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    s = torch.cuda.current_stream()
    s_out = torch.cuda.Stream()
    stream = ctypes.c_void_p(s.cuda_stream)
    h2d = sum(t.numel() * t.element_size() for t in (hx, hdz, hg, hb))
    d2h = sum(t.numel() * t.element_size() for t in outs)
    done = [torch.cuda.Event(), torch.cuda.Event()]    # step's kernels finished
    copied = [torch.cuda.Event(), torch.cuda.Event()]  # step's results copied out
    state = {"k": 0}

    def step():
        k = state["k"]
        P.x.copy_(hx, non_blocking=True)
        P.dz.copy_(hdz, non_blocking=True)
        P.gamma.copy_(hg, non_blocking=True)
        P.beta.copy_(hb, non_blocking=True)
        if k > 0:
            s.wait_event(copied[(k - 1) % 2])
        call(lib, fwd, stream)
        call(lib, bwd, stream)
        done[k % 2].record(s)
        s_out.wait_event(done[k % 2])
        with torch.cuda.stream(s_out):
            for d, h in zip(outs, houts):
                h.copy_(d, non_blocking=True)
        copied[k % 2].record(s_out)
        state["k"] = k + 1

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s)
    for _ in range(steps):
        step()
    s.wait_event(copied[(state["k"] - 1) % 2])   # the last copy-out is inside the region
    b.record(s)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    return {"value": round(step_bytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipelined": "copy-out of step k overlaps copy-in of step k + 1"}


def run_other_workloads(torch, rn, lib, rn_inputs, flush, peak, steps, warmup, only=None):
    """Full-size timing of the other workloads; ``only`` restricts the run to
    one group ("rms_small", "rms_current", "mxfp8", "large_fwd", "bwd_f32", "bwd_bf16",
    "rms_add", "moe_act")."""
    res = {}

    def want(name):
        return only is None or only == name

    def report(name, kind, N, H, esz, ln, ms, launches):
        b = algorithmic_bytes(kind, N, H, esz, ln)
        gbs = b / (ms * 1e-3) / 1e9
        res[name] = {"ms": round(ms, 5), "GBps": round(gbs, 1), "rows_per_s": round(N / (ms * 1e-3), 1),
                     "frac_of_peak": round(gbs / peak, 4), "pct_of_8TBps": round(gbs / 80.0, 2),
                     "algorithmic_bytes": b, "kernels_per_call": launches}

    if want("rms_small"):
        _small(torch, rn, lib, rn_inputs, flush, steps, warmup, report)
    if want("rms_current"):
        w = rn_inputs.make("rms_current")
        P = Prepared(rn, torch, w, ln=False)
        t = time_calls(torch, lib, [("cur", P.fwd_args("fp8_current"))], steps, warmup, flush)
        report("rms_16384x8192_fwd_fp8_current", "fwd_fp8_current", w.N, w.H, 2, False,
               statistics.mean(t["cur"]), 3)
        t = time_calls(torch, lib, [("nv", P.fwd_args("nvfp4"))], steps, warmup, flush)
        report("rms_16384x8192_fwd_nvfp4", "fwd_nvfp4", w.N, w.H, 2, False,
               statistics.mean(t["nv"]), 3)
        del P, w
    if want("mxfp8"):
        w = rn_inputs.make("mxfp8")
        for ln in (True, False):
            P = Prepared(rn, torch, w, ln=ln)
            t = time_calls(torch, lib, [("mx", P.fwd_args("mxfp8"))], steps, warmup, flush)
            report(f"{'ln' if ln else 'rms'}_65536x2048_fwd_mxfp8", "fwd_mxfp8", w.N, w.H, 2, ln,
                   statistics.mean(t["mx"]), 1)
            if ln:
                # the rowwise blocks alone (one pass of the row kernel)
                t = time_calls(torch, lib, [("mr", P.fwd_args("mxfp8_row"))], steps, warmup, flush)
                report("ln_65536x2048_fwd_mxfp8_rowwise_only", "fwd_mxfp8_row", w.N, w.H, 2, ln,
                       statistics.mean(t["mr"]), 1)
            del P
        del w
    if want("large_fwd"):
        # forward NONE and FP8 delayed at the largest shapes: the MXFP8
        # workload's rows (65536 x 2048, LayerNorm and RMSNorm) and the
        # current-scaling workload's (16384 x 8192, RMSNorm); the delayed
        # scale is a fixed 1.0 (the kernels' work does not depend on it)
        for wl, lns in (("mxfp8", (True, False)), ("rms_current", (False,))):
            w = rn_inputs.make(wl)
            for ln in lns:
                P = Prepared(rn, torch, w, ln=ln)
                tag = f"{'ln' if ln else 'rms'}_{w.N}x{w.H}"
                t = time_calls(torch, lib, [("n", P.fwd_args("none"))], steps, warmup, flush)
                report(f"{tag}_fwd_none", "fwd_none", w.N, w.H, 2, ln, statistics.mean(t["n"]), 1)
                t = time_calls(torch, lib, [("d", P.fwd_args("fp8_delayed", scale=1.0))], steps, warmup,
                               flush)
                report(f"{tag}_fwd_fp8_delayed", "fwd_fp8", w.N, w.H, 2, ln, statistics.mean(t["d"]), 2)
                del P
            del w
    if want("rms_small"):
        # the delayed-scaling history step (1024 entries): one tiny kernel,
        # launch-latency bound
        hist = torch.rand(1024, device="cuda")
        amax = torch.ones(1, device="cuda")
        scl = torch.ones(1, device="cuda")
        sinv = torch.empty(1, device="cuda")
        vp = ctypes.c_void_p
        fa = ("rn_delayed_scaling_update", [vp(hist.data_ptr()), 1024, vp(amax.data_ptr()),
                                            vp(scl.data_ptr()), vp(sinv.data_ptr())])
        t = time_calls(torch, lib, [("h", fa)], steps, warmup, flush)
        report("delayed_scaling_update_1024", "history", 1, 1024, 4, False, statistics.mean(t["h"]), 1)
    if want("rms_add"):
        w = rn_inputs.make("rms_add")
        P = Prepared(rn, torch, w, ln=False)
        t = time_calls(torch, lib, [("add", P.add_args("fp8_delayed", scale=w.scale))], steps, warmup,
                       flush)
        report("rms_add_8192x4096_fwd_fp8_delayed", "fwd_add_fp8", w.N, w.H, 2, False,
               statistics.mean(t["add"]), 2)
        # MXFP8 in both directions after the add: the row kernel (h, rowwise
        # blocks), then the two-direction kernel reading h back
        t = time_calls(torch, lib, [("addmx", P.add_args("mxfp8"))], steps, warmup, flush)
        report("rms_add_8192x4096_fwd_mxfp8", "fwd_add_mxfp8", w.N, w.H, 2, False,
               statistics.mean(t["addmx"]), 2)
        del P, w
    if want("moe_act"):
        # scaled SwiGLU of a mixture-of-experts MLP: 65536 tokens x 2048
        w = rn_inputs.make("moe_act")
        to = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to("cuda")
        x, dy = to(w.x), to(w.dz)
        sc = torch.from_numpy(w.scales).to("cuda")
        N, H = w.N, w.H
        vp, f32 = ctypes.c_void_p, ctypes.c_float
        keep = []

        def fwd_args(mode):
            o = rn._Output()
            if mode == "none":
                d = torch.empty((N, H), dtype=torch.bfloat16, device="cuda")
                o.data, o.out_dtype = d.data_ptr(), 0
                keep.append(d)
            elif mode == "fp8_current":
                d = torch.empty((N, H), dtype=torch.uint8, device="cuda")
                t3 = [torch.empty(1, dtype=torch.float32, device="cuda") for _ in range(3)]
                o.data, o.scale_out, o.scale_inv, o.amax = (d.data_ptr(), t3[0].data_ptr(),
                                                            t3[1].data_ptr(), t3[2].data_ptr())
                keep.extend([d] + t3)
            else:
                d = torch.empty((N, H), dtype=torch.uint8, device="cuda")
                r = torch.empty((N, H // 32), dtype=torch.uint8, device="cuda")
                o.data, o.row_scales = d.data_ptr(), r.data_ptr()
                keep.extend([d, r])
            keep.append(o)
            return ("rn_scaled_act_fwd", [1, vp(x.data_ptr()), 0, vp(sc.data_ptr()), N, H, f32(7.0),
                                          f32(1.702), rn.QUANT_MODES[mode], ctypes.byref(o)])

        dx = torch.empty_like(x)
        ds = torch.empty(N, dtype=torch.float32, device="cuda")
        bwd = ("rn_scaled_act_bwd", [1, vp(dy.data_ptr()), vp(x.data_ptr()), 0, vp(sc.data_ptr()), N, H,
                                     f32(7.0), f32(1.702), vp(dx.data_ptr()), vp(ds.data_ptr())])
        t = time_calls(torch, lib, [("none", fwd_args("none")), ("cur", fwd_args("fp8_current")),
                                    ("mx", fwd_args("mxfp8")), ("bwd", bwd)], steps, warmup, flush)
        report("swiglu_65536x2048_fwd_bf16", "act_fwd_none", N, H, 2, False, statistics.mean(t["none"]), 1)
        report("swiglu_65536x2048_fwd_fp8_current", "act_fwd_fp8_current", N, H, 2, False,
               statistics.mean(t["cur"]), 3)
        report("swiglu_65536x2048_fwd_mxfp8_rowwise", "act_fwd_mxfp8", N, H, 2, False,
               statistics.mean(t["mx"]), 1)
        report("swiglu_65536x2048_bwd", "act_bwd", N, H, 2, False, statistics.mean(t["bwd"]), 1)
        del x, dy, dx, keep, w
    for name in ("bwd_f32", "bwd_bf16"):
        if not want(name):
            continue
        w = rn_inputs.make(name)
        esz = 4 if w.dtype == "f32" else 2
        for ln in (True, False):
            P = Prepared(rn, torch, w, ln=ln)
            call(lib, P.fwd_args("none"), P.stream())      # mu / rsigma for the backward
            for margin in (0, 16):
                t = time_calls(torch, lib, [("b", P.bwd_args(margin))], steps, warmup, flush)
                report(f"{'ln' if ln else 'rms'}_{w.N}x{w.H}_{w.dtype}_bwd_margin{margin}", "bwd",
                       w.N, w.H, esz, ln, statistics.mean(t["b"]), 2)
            del P
        del w
    torch.cuda.synchronize()
    return res


def _small(torch, rn, lib, rn_inputs, flush, steps, warmup, report):
    w = rn_inputs.make("rms_small")
    P = Prepared(rn, torch, w, ln=False)
    calls = [("none", P.fwd_args("none"))]
    t = time_calls(torch, lib, calls, steps, warmup, flush)
    report("rms_256x1024_fwd_none", "fwd_none", w.N, w.H, 2, False, statistics.mean(t["none"]), 1)
    calls = [("dl", P.fwd_args("fp8_delayed", scale=w.scale)), ("bwd", P.bwd_args())]
    t = time_calls(torch, lib, calls, steps, warmup, flush)
    report("rms_256x1024_fwd_fp8_delayed", "fwd_fp8", w.N, w.H, 2, False, statistics.mean(t["dl"]), 1)
    report("rms_256x1024_bwd", "bwd", w.N, w.H, 2, False, statistics.mean(t["bwd"]), 2)
    del P


# ------------------------------------------------------- CPU oracle team
# The oracle on every host core: one spawned worker process per core (spawn,
# not fork: the parent may already hold a CUDA context), each regenerating
# the seeded workload once, untimed; a timed call deals row blocks to them.
_TEAM = {}


def _team_init(barrier, workload):
    import oracle
    import rn_inputs
    _TEAM["barrier"] = barrier
    _TEAM["w"] = rn_inputs.make(workload)
    _TEAM["oracle"] = oracle


def _team_sync(_):
    # every worker takes exactly one of these (each waits for all the others)
    _TEAM["barrier"].wait(timeout=900)
    return os.getpid()


def _team_block(rows):
    """LayerNorm fwd with FP8 delayed scaling + LayerNorm bwd of rows r0..r1
    of the ln_delayed workload, by the oracle as it stands."""
    r0, r1 = rows
    w, oracle = _TEAM["w"], _TEAM["oracle"]
    x = w.x_f64(slice(r0, r1))
    dz = w.dz_f64(slice(r0, r1))
    f = oracle.layernorm_fwd(x, w.gamma, w.beta, w.eps, True, "fp8_delayed", scale=w.scale)
    oracle.layernorm_bwd(dz, x, f["mu"], f["rsigma"], w.gamma, True, "bf16")
    return r1 - r0


class OracleTeam:
    """A pool of one oracle process per host core (numpy single-threaded in
    each: one worker per core is the parallelism)."""

    def __init__(self, workload="ln_delayed"):
        import multiprocessing as mp
        try:
            self.cores = len(os.sched_getaffinity(0))
        except AttributeError:
            self.cores = os.cpu_count() or 1
        ctx = mp.get_context("spawn")
        keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
        saved = {k: os.environ.get(k) for k in keys}
        for k in keys:
            os.environ[k] = "1"
        try:
            barrier = ctx.Barrier(self.cores)
            self.pool = ctx.Pool(self.cores, initializer=_team_init, initargs=(barrier, workload))
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        pids = self.pool.map(_team_sync, range(self.cores), chunksize=1)
        self.workers = len(set(pids))

    def run(self, r0, r1):
        """Rows r0..r1 in one block per worker; returns the wall seconds."""
        n = r1 - r0
        edges = [r0 + (n * i) // self.cores for i in range(self.cores + 1)]
        blocks = [(edges[i], edges[i + 1]) for i in range(self.cores) if edges[i + 1] > edges[i]]
        t0 = time.perf_counter()
        done = sum(self.pool.map(_team_block, blocks, chunksize=1))
        dt = time.perf_counter() - t0
        assert done == n
        return dt

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_baseline(w, step_bytes):
    """The oracle as it stands, on all host cores, over the whole headline
    workload once (fwd + FP8 delayed quantization + bwd), after a warm-up
    over one small block a core."""
    team = OracleTeam("ln_delayed")
    try:
        team.run(0, min(w.N, 8 * team.cores))
        dt = team.run(0, w.N)
    finally:
        team.close()
    return {"value": round(step_bytes / dt / 1e9, 4), "unit": "GB/s", "cores": team.cores,
            "workers": team.workers, "kind": "oracle",
            "rows_per_s": round(w.N / dt, 1),
            "sample": f"the full workload, {w.N} rows x {w.H}, one fwd+bwd pass ({dt:.2f} s wall on "
                      f"{team.cores} cores; numpy fp64, one process a core, row blocks)"}


# ---------------------------------------------------------- reference arm
def run_reference(args):
    """The oracle (the only reference this method has here) on all host
    cores; each step is a bounded sample of the headline workload: 64 rows
    a core, the next rows each step."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import rn_inputs
    w = rn_inputs.make("ln_delayed")
    team = OracleTeam("ln_delayed")
    rows = min(w.N, 64 * team.cores)
    per_sample = algorithmic_bytes("fwd_fp8", rows, w.H, 2, True) + algorithmic_bytes("bwd", rows, w.H, 2, True)

    def step(k):
        r0 = (k * rows) % w.N
        r0 = min(r0, w.N - rows)
        return team.run(r0, r0 + rows)

    try:
        for k in range(args.warmup):
            step(k)
        times = [step(args.warmup + k) for k in range(args.steps)]
    finally:
        team.close()
    dt = sum(times) / len(times)
    v = per_sample / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded rn_inputs workload ln_delayed)",
            "config": {"workload": "LayerNorm fwd (FP8 delayed) + bwd, bf16 [8192 x 4096], "
                                   f"each step a {rows}-row sample",
                       "rows_per_s": round(rows / dt, 1)},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": team.cores,
                             "workers": team.workers, "kind": "oracle",
                             "sample": f"{rows} consecutive rows of 8192 per step ({rows // team.cores} "
                                       "a core), one process a core"},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="rn", choices=["rn", "reference"])
    ap.add_argument("--quick", action="store_true", help="headline workload only")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--only", default=None,
                    choices=["rms_small", "rms_current", "mxfp8", "large_fwd", "bwd_f32", "bwd_bf16",
                             "rms_add", "moe_act"],
                    help="time only this workload group (prints its results; for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_rn(args)


if __name__ == "__main__":
    main()
