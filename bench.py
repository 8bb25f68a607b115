#!/usr/bin/env python
"""Benchmark: attention TFLOP/s (forward and forward+backward, bf16) on GB300.

One step = the whole training-direction hot path on the headline workload
(B=4, H=32, N=4096, d=128, non-causal, bf16 inputs drawn i.i.d. N(0,1) from a seed):
fa_fwd, then fa_bwd_prep, fa_bwd_main, fa_bwd_finish (the three steps of fa_bwd).
``value`` = algorithmic forward+backward FLOP of all ranks / max-over-ranks time.

Also measured in the same run and reported in the same JSON line:
  breakdown.fwd            forward alone, same workload
  breakdown.*_causal       the causal variant of the workload
  breakdown.decode         split-KV decode (B=64, H=32, N_kv=32768, d=128, 64 splits), GB/s
  breakdown.decode_paged   the same decode over a paged cache (256-key blocks, shuffled), GB/s
  breakdown.fwd_fp8*       forward from e4m3 Q, K, V (per-tensor scales), same shapes; the
                           fraction is of the fp8 GEMM rate measured in the same run
  breakdown.gemm_peaks     dense 8192^3 GEMM rates measured here (torch.matmul bf16 and
                           torch._scaled_mm e4m3, best of 10): the fp8 denominator
  breakdown.gpt2m_*        a GPT-2-medium attention layer, 8x16x1024x64 causal, fwd and fwd+bwd;
                           its inputs fit in L2, so a 256 MB buffer is written before every
                           timed call; per-call CUDA events
  breakdown.long_*         1x16x16384x128 causal with outlier keys, fwd and fwd+bwd
  breakdown.window         forward and forward+backward under a 4096-key causal sliding window
                           (left 4095, right 0) on 1x16x16384x128
  breakdown.block_sparse   the same shape under a causal 128x128 block pattern (a band of one
                           block, the first key block, 5% random blocks; ``density`` = share of
                           blocks set); FLOP = 4 d (fwd), 10 d (bwd) per visible pair
  breakdown.varlen         a packed batch of 16 causal sequences of 512..8192 tokens (seed
                           1006, H=32, d=128), forward and forward+backward
  roofline                 the dominant kernel of the step (backward main kernel), timed alone
  e2e                      the step through the public Python API with host (pinned) buffers,
                           host->device and device->host copies inside the timed region
  cpu_baseline             the fp64 oracle on a bounded sample, on this machine's host cores
  clocks                   nvidia-smi samples taken while the timed regions ran
  summary                  (last key of the line) [rate, fraction of measured peak] per workload

``--impl reference`` times the fp64 CPU oracle instead (the reference arm for this build).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Multi-GPU (one process per GPU): torchrun --nproc-per-node N bench.py --gpus N ...
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention TFLOP/s fwd & fwd+bwd (bf16, causal/non) and % of GB300 BF16 peak"
UNIT = "TFLOP/s"
# Measured GB300 denominators (this pool): used when MEASURED_PEAKS.json is absent.
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


# ---------------------------------------------------------------------------------------------
# small helpers (host logic, testable without a GPU)
# ---------------------------------------------------------------------------------------------

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def whole_job_rate(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Aggregate throughput: the units all ranks processed / the slowest rank's time."""
    return units_per_rank * world / max_seconds


def reduce_max(x: float) -> float:
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        import torch
        dev = "cuda" if (dist.get_backend() == "nccl") else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return x


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def source_digest(*rel_paths) -> str:
    h = hashlib.sha256()
    for rp in rel_paths:
        with open(os.path.join(ROOT, rp), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key: str, digest: str):
    """DRAM bytes per launch from the committed ncu summary, or None if the kernel changed."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e or e.get("source_digest") != digest:
        return None
    return e.get("dram_bytes_per_launch")


def parse_clock_csv(text: str):
    """Summarise nvidia-smi CSV samples: median SM MHz under load, max MHz, active reasons."""
    rows = [r.strip() for r in text.strip().splitlines() if r.strip()]
    if len(rows) < 2:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    hdr = [h.strip() for h in rows[0].split(",")]
    recs = []
    for r in rows[1:]:
        cols = [c.strip() for c in r.split(",")]
        if len(cols) != len(hdr):
            continue
        recs.append(dict(zip(hdr, cols)))

    def num(s):
        try:
            return float(s.split()[0])
        except (ValueError, IndexError):
            return None

    sm = [num(r.get("clocks.current.sm [MHz]", r.get("clocks.sm [MHz]", ""))) for r in recs]
    mx = [num(r.get("clocks.max.sm [MHz]", "")) for r in recs]
    pw = [num(r.get("power.draw [W]", "")) for r in recs]
    loaded = [s for s, p in zip(sm, pw) if s is not None and p is not None and p > 250.0]
    reasons = set()
    for r in recs:
        for key in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"):
            for k, v in r.items():
                if k.startswith("clocks_event_reasons." + key) and v.strip().lower() == "active":
                    reasons.add(key)
    return {
        "sm_mhz": statistics.median(loaded) if loaded else (statistics.median([s for s in sm if s]) if any(sm) else None),
        "sm_max_mhz": max([m for m in mx if m], default=None),
        "reasons": sorted(reasons),
        "samples": len(recs),
        "samples_under_load": len(loaded),
    }


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.path = os.path.join("/tmp", f"fa_bench_clocks_{os.getpid()}.csv")
        self.gpu_id = gpu_id

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv", "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        with open(self.path) as f:
            text = f.read()
        os.unlink(self.path)
        return parse_clock_csv(text)


# ---------------------------------------------------------------------------------------------
# CPU oracle timing (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------------------------

def oracle_sample_step(x, heads, w):
    """fp64 oracle forward + backward for the listed (b, h) heads; returns algorithmic FLOP."""
    from oracle import attention as A
    from exact_io_aware_08_gb300 import accounting as W
    flop = 0
    for b, h in heads:
        A.forward_head(x["q"][b, h], x["k"][b, h], x["v"][b, h], w.scale, w.causal)
        A.backward_head(x["q"][b, h], x["k"][b, h], x["v"][b, h], x["do"][b, h], w.scale, w.causal)
        flop += W.fwd_flops(1, 1, w.N_q, w.N_kv, w.d, w.causal) + W.bwd_flops(1, 1, w.N_q, w.N_kv, w.d, w.causal)
    return flop


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def head_sample_inputs(w, n_heads):
    """fp64 copies of the first n_heads heads of the workload (same seeded draw)."""
    import torch
    from exact_io_aware_08_gb300 import inputs
    x = inputs.make_workload(w)
    out = {}
    for k, t in x.items():
        out[k] = t.reshape(w.B * w.H, t.shape[2], t.shape[3])[:n_heads].to(torch.float64).numpy()
    return {k: v[:, None] for k, v in out.items()}   # [n, 1, N, d]


def time_oracle(w, budget_s: float = 12.0, max_heads: int = 8):
    """Time the oracle on whole heads of the workload until ~budget_s; returns dict."""
    x = head_sample_inputs(w, max_heads)
    done, flop, t0 = 0, 0, time.perf_counter()
    while done < max_heads:
        flop += oracle_sample_step(x, [(done, 0)], w)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {
        "value": flop / dt / 1e12, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
        "sample": f"fp64 NumPy oracle, forward+backward of {done} whole head(s) of {w.name} "
                  f"(explicit N x N score matrix), {dt:.1f} s wall; algorithmic FLOP counted",
    }


def summarize(bd, peak_tf):
    """Compact per-workload figures: [TFLOP/s (GB/s for decode), fraction of its peak]."""
    def pair(rate, frac):
        return [rate, None if frac is None else round(frac, 3)]

    def tf(name, key="tflops"):
        e = bd.get(name) or {}
        v = e.get(key)
        return pair(v, None if v is None else v / peak_tf)
    out = {"unit": "[TFLOP/s or GB/s, frac of measured peak]",
           "fwd": pair(bd["fwd"]["tflops"], bd["fwd"]["frac_of_peak"]),
           "fwd_bwd": tf("fwd_bwd"), "fwd_causal": tf("fwd_causal"), "fwd_bwd_causal": tf("fwd_bwd_causal")}
    for name in ("gpt2m_8x16x1024x64_causal", "long_1x16x16384x128_causal_outliers"):
        e = bd.get(name)
        if e:
            short = "gpt2m" if name.startswith("gpt2m") else "long"
            out[short + "_fwd"] = pair(e["fwd_tflops"], e.get("fwd_frac"))
            out[short + "_fwd_bwd"] = pair(e["fwd_bwd_tflops"], e.get("fwd_bwd_frac"))
    for name in ("window", "block_sparse", "varlen"):
        if name in bd:
            out[name + "_fwd_bwd"] = tf(name, "fwd_bwd_tflops")
    for name in ("fwd_fp8", "fwd_fp8_causal"):
        if name in bd:
            out[name] = pair(bd[name]["tflops"], bd[name]["frac_of_fp8_peak"])
    if "gemm_peaks" in bd:
        out["fp8_peak"] = bd["gemm_peaks"].get("fp8_peak_used")
    for name in ("decode", "decode_paged"):
        if name in bd:
            out[name] = pair(bd[name]["gbps"], bd[name]["frac_of_hbm"])
    return out


def measure_gemm_peaks(dev, n=8192, reps=10):
    """Dense GEMM rates on this GPU, timed the way the bf16 peak was: n^3 products, 2 n^3 FLOP,
    best of ``reps`` CUDA-event timings after warm-up.  fp8 is torch._scaled_mm on e4m3 inputs
    (unit scales, bf16 out); bf16 is torch.matmul, for the fp8 : bf16 ratio on the same box."""
    import torch
    out = {"n": n}

    def best_ms(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(reps):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            fn()
            e.record()
            e.synchronize()
            best = min(best, s.elapsed_time(e))
        return best
    flop = 2.0 * n ** 3
    a = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    b = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    out["bf16_tflops_measured"] = round(flop / (best_ms(lambda: a @ b) * 1e-3) / 1e12, 1)
    try:
        a8 = a.to(torch.float8_e4m3fn)
        b8 = b.to(torch.float8_e4m3fn).t()                # column-major second operand
        one = torch.ones((), device=dev, dtype=torch.float32)
        ms = best_ms(lambda: torch._scaled_mm(a8, b8, scale_a=one, scale_b=one, out_dtype=torch.bfloat16))
        out["fp8_tflops_measured"] = round(flop / (ms * 1e-3) / 1e12, 1)
    except (RuntimeError, AttributeError, TypeError) as ex:   # no fp8 GEMM in this torch build
        out["fp8_error"] = str(ex).splitlines()[0][:120]
    del a, b
    return out


# ---------------------------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------------------------

def run_ours(args, rank, world, local_rank):
    import torch
    import exact_io_aware_08_gb300 as fa
    from exact_io_aware_08_gb300 import accounting as W
    from exact_io_aware_08_gb300 import build as fabuild
    from exact_io_aware_08_gb300 import inputs

    fabuild.build()
    fa.load_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    peak_tf = peaks["bf16_tflops"]
    peak_hbm = peaks["hbm_gbs"]
    stream = torch.cuda.current_stream()
    K, Wm = args.steps, args.warmup

    def ev():
        return torch.cuda.Event(enable_timing=True)

    # ---------------------------------------------------------------- headline workloads
    def setup(w):
        x = inputs.make_qkv(w.B, w.H, w.N_q, w.N_kv, w.d, w.seed + 7919 * rank)
        d = {k: v.to(dev) for k, v in x.items()}
        d["o"] = torch.empty_like(d["q"])
        d["lse"] = torch.empty(d["q"].shape[:3], dtype=torch.float32, device=dev)
        d["dq"] = torch.empty_like(d["q"])
        d["dk"] = torch.empty_like(d["k"])
        d["dv"] = torch.empty_like(d["v"])
        d["ws"] = torch.empty(fa.fa_bwd_workspace_size(w.B, w.H, w.N_q, w.N_kv, w.d),
                              dtype=torch.uint8, device=dev)
        return x, d

    def fwd(w, d):
        fa.fa_fwd(d["q"], d["k"], d["v"], d["o"], d["lse"], w.scale, w.causal)

    def bwd(w, d, main_events=None):
        fa.fa_bwd_prep(d["o"], d["do"], d["ws"], w.N_kv)
        if main_events is not None:
            main_events[0].record(stream)
        fa.fa_bwd_main(d["q"], d["k"], d["v"], d["lse"], d["do"], d["dk"], d["dv"], d["ws"],
                       w.scale, w.causal)
        if main_events is not None:
            main_events[1].record(stream)
        fa.fa_bwd_finish(d["dq"], d["ws"], w.N_kv, w.scale)

    def nvtx(push, label=None):
        """NVTX range markers; a no-op where this torch build has none."""
        try:
            if push:
                torch.cuda.nvtx.range_push(label)
            else:
                torch.cuda.nvtx.range_pop()
        except (AttributeError, RuntimeError):
            pass

    def timed(fn, steps, inner=False, name=None):
        """Warm up, then time ``steps`` calls between barriers; optional per-call events.  The
        timed region is an NVTX range (named after the timed function) for profiler timelines."""
        for _ in range(Wm):
            fn(None)
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        s, e = ev(), ev()
        nvtx(True, name or getattr(fn, "__name__", "timed"))
        s.record(stream)
        per = []
        for _ in range(steps):
            pe = (ev(), ev()) if inner else None
            fn(pe)
            if inner:
                per.append(pe)
        e.record(stream)
        nvtx(False)
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        return s.elapsed_time(e), [a.elapsed_time(b) for a, b in per]

    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
    smi_index = vis[local_rank] if len(vis) > local_rank and vis[local_rank].strip().isdigit() else str(local_rank)
    sampler = ClockSampler(smi_index)
    w = inputs.HEADLINE
    wc = inputs.HEADLINE_CAUSAL
    x, d = setup(w)
    fl_f = W.fwd_flops(w.B, w.H, w.N_q, w.N_kv, w.d, w.causal)
    fl_b = W.bwd_flops(w.B, w.H, w.N_q, w.N_kv, w.d, w.causal)

    sampler.start()
    # ---- the step: fwd + bwd (F1, F2, F3, F4); F3 bracketed by events
    def step(pe):
        fwd(w, d)
        bwd(w, d, pe)
    total_ms, main_ms = timed(step, K, inner=True)
    ms_step = reduce_max(total_ms / K)
    value = whole_job_rate(fl_f + fl_b, world, ms_step * 1e-3) / 1e12
    bwd_main_ms = statistics.mean(main_ms)
    achieved = fl_b / (bwd_main_ms * 1e-3) / 1e12
    digest = source_digest("exact_io_aware_08_gb300/csrc/bwd.cu", "exact_io_aware_08_gb300/csrc/sm103.cuh")
    roofline = {
        "bound": "tensor", "achieved": round(achieved, 1), "peak": peak_tf, "unit": "TFLOP/s",
        "frac": round(achieved / peak_tf, 4),
        "traffic": profiled_traffic("bwd_main_kernel<128>", digest),
        "kernel": "fa::bwd_main_kernel<128> (F3)",
        "work_per_launch": f"{fl_b:.4e} FLOP (10*d*N_q*N_kv*B*H)",
        "avg_launch_ms": round(bwd_main_ms, 4),
        "peak_source": f"bf16_tflops (burst), {peak_src}",
    }

    # ---- forward alone (F1 timed alone: one kernel per call)
    def fwd_only(pe):
        if pe is not None:
            pe[0].record(stream)
        fwd(w, d)
        if pe is not None:
            pe[1].record(stream)
    f_total, f_inner = timed(fwd_only, K, inner=True)
    f_ms = reduce_max(f_total / K)
    fwd_kernel_ms = statistics.mean(f_inner)
    breakdown = {
        "fwd": {"tflops": round(whole_job_rate(fl_f, world, f_ms * 1e-3) / 1e12, 1),
                "ms": round(f_ms, 4), "frac_of_peak": round(fl_f / (fwd_kernel_ms * 1e-3) / 1e12 / peak_tf, 4),
                "kernel_ms": round(fwd_kernel_ms, 4)},
        "fwd_bwd": {"tflops": round(value, 1), "ms": round(ms_step, 4),
                    "frac_of_peak": round(value / world / peak_tf, 4)},
    }
    # ---- causal variant (shares buffers: same shapes)
    xc = inputs.make_qkv(wc.B, wc.H, wc.N_q, wc.N_kv, wc.d, wc.seed + 7919 * rank)
    for k_ in ("q", "k", "v", "do"):
        d[k_].copy_(xc[k_])
    del xc
    fl_fc = W.fwd_flops(wc.B, wc.H, wc.N_q, wc.N_kv, wc.d, True)
    fl_bc = W.bwd_flops(wc.B, wc.H, wc.N_q, wc.N_kv, wc.d, True)
    c_total, _ = timed(lambda pe: (fwd(wc, d), bwd(wc, d)), K)
    cf_total, _ = timed(lambda pe: fwd(wc, d), K)
    c_ms, cf_ms = reduce_max(c_total / K), reduce_max(cf_total / K)
    breakdown["fwd_bwd_causal"] = {"tflops": round(whole_job_rate(fl_fc + fl_bc, world, c_ms * 1e-3) / 1e12, 1),
                                   "ms": round(c_ms, 4)}
    breakdown["fwd_causal"] = {"tflops": round(whole_job_rate(fl_fc, world, cf_ms * 1e-3) / 1e12, 1),
                               "ms": round(cf_ms, 4)}

    # ---- the other two training-direction workloads: a GPT-2-medium layer (8x16x1024x64,
    # causal) and the long causal sequence with outlier keys (1x16x16384x128)
    l2_flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for wx in (inputs.GPT2M, inputs.LONG):
        xx = {k_: v_.to(dev) for k_, v_ in inputs.make_workload(wx).items()}
        ox, lx = torch.empty_like(xx["q"]), torch.empty(xx["q"].shape[:3], dtype=torch.float32, device=dev)
        gx = [torch.empty_like(xx["q"]) for _ in range(3)]
        wsx = torch.empty(fa.fa_bwd_workspace_size(wx.B, wx.H, wx.N_q, wx.N_kv, wx.d), dtype=torch.uint8,
                          device=dev)
        flx_f = W.fwd_flops(wx.B, wx.H, wx.N_q, wx.N_kv, wx.d, wx.causal)
        flx_b = W.bwd_flops(wx.B, wx.H, wx.N_q, wx.N_kv, wx.d, wx.causal)

        small = wx is inputs.GPT2M       # its inputs fit in L2: flush before every timed call

        def fx(pe, wx=wx, xx=xx, ox=ox, lx=lx, small=small):
            if small:
                l2_flush.zero_()
            if pe is not None:
                pe[0].record(stream)
            fa.fa_fwd(xx["q"], xx["k"], xx["v"], ox, lx, wx.scale, wx.causal)
            if pe is not None:
                pe[1].record(stream)

        def fbx(pe, wx=wx, xx=xx, ox=ox, lx=lx, gx=gx, wsx=wsx, small=small):
            if small:
                l2_flush.zero_()
            if pe is not None:
                pe[0].record(stream)
            fa.fa_fwd(xx["q"], xx["k"], xx["v"], ox, lx, wx.scale, wx.causal)
            fa.fa_bwd(xx["q"], xx["k"], xx["v"], ox, lx, xx["do"], gx[0], gx[1], gx[2], wsx, wx.scale,
                      wx.causal)
            if pe is not None:
                pe[1].record(stream)
        _, tf = timed(fx, K, inner=True)
        _, tfb = timed(fbx, K, inner=True)
        mf, mfb = reduce_max(statistics.mean(tf)), reduce_max(statistics.mean(tfb))
        breakdown[wx.name] = {
            "fwd_tflops": round(whole_job_rate(flx_f, world, mf * 1e-3) / 1e12, 1), "fwd_ms": round(mf, 4),
            "fwd_bwd_tflops": round(whole_job_rate(flx_f + flx_b, world, mfb * 1e-3) / 1e12, 1),
            "fwd_bwd_ms": round(mfb, 4),
            "fwd_frac": round(flx_f / (mf * 1e-3) / 1e12 / peak_tf, 4),
            "fwd_bwd_frac": round((flx_f + flx_b) / (mfb * 1e-3) / 1e12 / peak_tf, 4),
        }
        del xx, ox, lx, gx, wsx
    del l2_flush

    # ---- sliding window on the long sequence: 1x16x16384x128, each query sees its last 4096 keys
    wl_ = inputs.LONG
    win = 4095
    xw = {k_: v_.to(dev) for k_, v_ in inputs.make_workload(wl_).items()}
    ow, lw = torch.empty_like(xw["q"]), torch.empty(xw["q"].shape[:3], dtype=torch.float32, device=dev)
    gw = [torch.empty_like(xw["q"]) for _ in range(3)]
    wsw = torch.empty(fa.fa_bwd_workspace_size(wl_.B, wl_.H, wl_.N_q, wl_.N_kv, wl_.d), dtype=torch.uint8,
                      device=dev)
    fl_wf = W.window_fwd_flops(wl_.B, wl_.H, wl_.N_q, wl_.d, win, 0)
    fl_wb = W.window_bwd_flops(wl_.B, wl_.H, wl_.N_q, wl_.d, win, 0)

    def win_fwd(pe):
        fa.fa_fwd_window(xw["q"], xw["k"], xw["v"], ow, lw, wl_.scale, win, 0)

    def win_step(pe):
        win_fwd(pe)
        fa.fa_bwd_window(xw["q"], xw["k"], xw["v"], ow, lw, xw["do"], gw[0], gw[1], gw[2], wsw,
                         wl_.scale, win, 0)
    wf_total, _ = timed(win_fwd, K)
    ws_total, _ = timed(win_step, K)
    wf_ms, ws_ms = reduce_max(wf_total / K), reduce_max(ws_total / K)
    breakdown["window"] = {
        "fwd_tflops": round(whole_job_rate(fl_wf, world, wf_ms * 1e-3) / 1e12, 1), "fwd_ms": round(wf_ms, 4),
        "fwd_bwd_tflops": round(whole_job_rate(fl_wf + fl_wb, world, ws_ms * 1e-3) / 1e12, 1),
        "fwd_bwd_ms": round(ws_ms, 4),
    }
    # ---- block-sparse on the same long sequence: 128 x 128 blocks, a band of one block either
    # side of the diagonal, the first key block and 5% random blocks, causal inside the blocks
    bmask = inputs.make_block_mask(-(-wl_.N_q // fa.BLOCK_SIZE), -(-wl_.N_kv // fa.BLOCK_SIZE), 1005)
    bpairs = W.block_sparse_pairs(bmask, wl_.N_q, wl_.N_kv, True) * wl_.B * wl_.H
    bmask_d = bmask.to(dev)
    fl_bf, fl_bb = 4 * wl_.d * bpairs, 10 * wl_.d * bpairs

    def bs_fwd(pe):
        fa.fa_fwd_block_sparse(xw["q"], xw["k"], xw["v"], ow, lw, wl_.scale, bmask_d, True)

    def bs_step(pe):
        bs_fwd(pe)
        fa.fa_bwd_block_sparse(xw["q"], xw["k"], xw["v"], ow, lw, xw["do"], gw[0], gw[1], gw[2], wsw,
                               wl_.scale, bmask_d, True)
    bf_total, _ = timed(bs_fwd, K)
    bb_total, _ = timed(bs_step, K)
    bf_ms, bb_ms = reduce_max(bf_total / K), reduce_max(bb_total / K)
    breakdown["block_sparse"] = {
        "density": round(float(bmask.float().mean()), 4),
        "fwd_tflops": round(whole_job_rate(fl_bf, world, bf_ms * 1e-3) / 1e12, 1), "fwd_ms": round(bf_ms, 4),
        "fwd_bwd_tflops": round(whole_job_rate(fl_bf + fl_bb, world, bb_ms * 1e-3) / 1e12, 1),
        "fwd_bwd_ms": round(bb_ms, 4),
    }
    del xw, ow, lw, gw, wsw, bmask_d

    # ---- variable-length batch: 16 packed causal sequences of 512..8192 tokens, 32 heads, d=128
    vlens = inputs.make_varlen_lengths(16, 512, 8192, 1006)
    vH, vd = 32, 128
    vtot = sum(vlens)
    xv = inputs.make_packed(vtot, vH, vd, 1006 + 7919 * rank, device=str(dev))
    vcu = torch.tensor([sum(vlens[:i]) for i in range(len(vlens) + 1)], dtype=torch.int32, device=dev)
    vmax = max(vlens)
    ov = torch.empty_like(xv["q"])
    lv = torch.empty((vH, vtot), dtype=torch.float32, device=dev)
    gv = [torch.empty_like(xv["q"]) for _ in range(3)]
    wsv = torch.empty(fa.fa_bwd_workspace_size(1, vH, vtot, vtot, vd), dtype=torch.uint8, device=dev)
    vpairs = sum(W.pairs(n_, n_, True) for n_ in vlens) * vH
    fl_vf, fl_vb = 4 * vd * vpairs, 10 * vd * vpairs
    vscale = vd ** -0.5

    def vl_fwd(pe):
        fa.fa_fwd_varlen(xv["q"], xv["k"], xv["v"], ov, lv, vcu, vcu, vmax, vmax, vscale, True)

    def vl_step(pe):
        vl_fwd(pe)
        fa.fa_bwd_varlen(xv["q"], xv["k"], xv["v"], ov, lv, xv["do"], gv[0], gv[1], gv[2], wsv, vcu, vcu,
                         vmax, vmax, vscale, True)
    vf_total, _ = timed(vl_fwd, K)
    vb_total, _ = timed(vl_step, K)
    vf_ms, vb_ms = reduce_max(vf_total / K), reduce_max(vb_total / K)
    breakdown["varlen"] = {
        "tokens": vtot,
        "fwd_tflops": round(whole_job_rate(fl_vf, world, vf_ms * 1e-3) / 1e12, 1), "fwd_ms": round(vf_ms, 4),
        "fwd_bwd_tflops": round(whole_job_rate(fl_vf + fl_vb, world, vb_ms * 1e-3) / 1e12, 1),
        "fwd_bwd_ms": round(vb_ms, 4),
    }
    del xv, ov, lv, gv, wsv

    # ---- FP8 forward (e4m3 Q, K, V with per-tensor scales) on the same shapes
    x8 = inputs.make_qkv_fp8(w.B, w.H, w.N_q, w.N_kv, w.d, w.seed + 7919 * rank, device=str(dev))
    gemm = measure_gemm_peaks(dev)
    if gemm.get("fp8_tflops_measured"):
        peak_f8, peak_f8_src = gemm["fp8_tflops_measured"], "measured e4m3 GEMM, this run"
    else:
        peak_f8, peak_f8_src = 2 * peak_tf, "2 x bf16_tflops (nominal ratio; fp8 GEMM unavailable)"

    def fwd8(causal):
        def f(pe):
            if pe is not None:
                pe[0].record(stream)
            fa.fa_fwd_fp8(x8["q8"], x8["k8"], x8["v8"], d["o"], d["lse"], w.scale, x8["descale_q"],
                          x8["descale_k"], x8["descale_v"], causal)
            if pe is not None:
                pe[1].record(stream)
        return f
    for causal, key, fl in ((False, "fwd_fp8", fl_f), (True, "fwd_fp8_causal", fl_fc)):
        t8, i8 = timed(fwd8(causal), K, inner=True)
        ms8 = reduce_max(t8 / K)
        k8 = statistics.mean(i8)
        breakdown[key] = {"tflops": round(whole_job_rate(fl, world, ms8 * 1e-3) / 1e12, 1),
                          "ms": round(ms8, 4), "kernel_ms": round(k8, 4),
                          "frac_of_fp8_peak": round(fl / (k8 * 1e-3) / 1e12 / peak_f8, 4),
                          "traffic": profiled_traffic("fwd_kernel<128, fp8>", source_digest(
                              "exact_io_aware_08_gb300/csrc/fwd.cu", "exact_io_aware_08_gb300/csrc/sm103.cuh"))
                          if not causal else None}
    del x8
    breakdown["gemm_peaks"] = dict(gemm, fp8_peak_used=round(peak_f8, 1), fp8_peak_source=peak_f8_src)

    # ---- e2e through the public API with pinned host buffers (restore the headline inputs)
    host = {k_: x[k_].pin_memory() for k_ in ("q", "k", "v", "do")}
    out_host = {
        "o": torch.empty(x["q"].shape, dtype=torch.bfloat16).pin_memory(),
        "lse": torch.empty(x["q"].shape[:3], dtype=torch.float32).pin_memory(),
        "dq": torch.empty(x["q"].shape, dtype=torch.bfloat16).pin_memory(),
        "dk": torch.empty(x["k"].shape, dtype=torch.bfloat16).pin_memory(),
        "dv": torch.empty(x["v"].shape, dtype=torch.bfloat16).pin_memory(),
    }
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in out_host.values())

    # Pipelined like a training input loop: step i+1's inputs go host->device on one copy stream
    # while step i computes, and step i's outputs go device->host on another (o and lse as soon
    # as the forward ends, the gradients after the backward).  Inputs and outputs rotate through
    # three device buffer sets; every step's copies fall inside the timed region.
    cs = stream
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    NSL = 3                                  # device buffer sets in flight
    dbuf = [{k_: torch.empty_like(d[k_]) for k_ in ("q", "k", "v", "do")} for _ in range(NSL)]
    dout = [{"o": torch.empty_like(d["q"]), "lse": torch.empty_like(d["lse"]), "dq": torch.empty_like(d["q"]),
             "dk": torch.empty_like(d["k"]), "dv": torch.empty_like(d["v"])} for _ in range(NSL)]
    in_ready = [torch.cuda.Event() for _ in range(NSL)]
    in_free = [torch.cuda.Event() for _ in range(NSL)]
    fwd_done = [torch.cuda.Event() for _ in range(NSL)]
    bwd_done = [torch.cuda.Event() for _ in range(NSL)]
    out_free = [torch.cuda.Event() for _ in range(NSL)]

    def issue_h2d(i):
        sl = i % NSL
        with torch.cuda.stream(s_in):
            if i >= NSL:
                s_in.wait_event(in_free[sl])
            for k_ in ("q", "k", "v", "do"):
                dbuf[sl][k_].copy_(host[k_], non_blocking=True)
            in_ready[sl].record(s_in)

    def e2e_run(n_steps):
        issue_h2d(0)
        for i in range(n_steps):
            sl = i % NSL
            if i + 1 < n_steps:
                issue_h2d(i + 1)
            b, o = dbuf[sl], dout[sl]
            cs.wait_event(in_ready[sl])
            if i >= NSL:
                cs.wait_event(out_free[sl])
            fa.fa_fwd(b["q"], b["k"], b["v"], o["o"], o["lse"], w.scale, w.causal, cs)
            fwd_done[sl].record(cs)
            fa.fa_bwd(b["q"], b["k"], b["v"], o["o"], o["lse"], b["do"], o["dq"], o["dk"], o["dv"], d["ws"],
                      w.scale, w.causal, cs)
            in_free[sl].record(cs)
            bwd_done[sl].record(cs)
            with torch.cuda.stream(s_out):
                s_out.wait_event(fwd_done[sl])
                out_host["o"].copy_(o["o"], non_blocking=True)
                out_host["lse"].copy_(o["lse"], non_blocking=True)
                s_out.wait_event(bwd_done[sl])
                for k_ in ("dq", "dk", "dv"):
                    out_host[k_].copy_(o[k_], non_blocking=True)
                out_free[sl].record(s_out)
        cs.wait_stream(s_out)
        cs.wait_stream(s_in)

    e2e_run(Wm)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    es, ee = ev(), ev()
    es.record(cs)
    e2e_run(K)
    ee.record(cs)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    e_ms = reduce_max(es.elapsed_time(ee) / K)
    e2e = {"value": round(whole_job_rate(fl_f + fl_b, world, e_ms * 1e-3) / 1e12, 1), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e_ms, 4),
           "api": "fa_fwd + fa_bwd (C ABI), pinned host buffers, 3 device buffer sets"}
    del dbuf, dout
    del d, x, host, out_host
    torch.cuda.empty_cache()

    # ---- split-KV decode (F5 + F6), HBM-bound
    wd = inputs.DECODE
    xd = inputs.make_workload(wd, with_do=False, device=str(dev))
    od = torch.empty_like(xd["q"])
    lsed = torch.empty((wd.B, wd.H, 1), dtype=torch.float32, device=dev)
    wsd = torch.empty(fa.fa_decode_workspace_size(wd.B, wd.H, wd.N_kv, wd.d, wd.n_splits),
                      dtype=torch.uint8, device=dev)

    def dec(pe):
        if pe is not None:
            pe[0].record(stream)
        fa.fa_decode_splitkv(xd["q"], xd["k"], xd["v"], od, lsed, wd.scale, wd.n_splits, wsd)
        if pe is not None:
            pe[1].record(stream)
    dk_total, dk_inner = timed(dec, K, inner=True)
    dec_ms = reduce_max(dk_total / K)
    bytes_dec = W.decode_bytes(wd.B, wd.H, wd.N_kv, wd.d)
    part = W.decode_partial_bytes(wd.B, wd.H, wd.d, wd.n_splits)
    gbs = bytes_dec / (statistics.mean(dk_inner) * 1e-3) / 1e9
    breakdown["decode"] = {
        "gbps": round(whole_job_rate(bytes_dec, world, dec_ms * 1e-3) / 1e9, 1),
        "ms": round(dec_ms, 4), "frac_of_hbm": round(gbs / peak_hbm, 4),
        "gbps_incl_partials": round((bytes_dec + part) / (statistics.mean(dk_inner) * 1e-3) / 1e9, 1),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak_hbm, "unit": "GB/s",
                     "frac": round(gbs / peak_hbm, 4),
                     "traffic": profiled_traffic("decode_split_kernel<128>", source_digest(
                         "exact_io_aware_08_gb300/csrc/decode.cu", "exact_io_aware_08_gb300/csrc/sm103.cuh")),
                     "work_per_launch": bytes_dec},
    }

    # ---- the same decode over a paged cache: 256-key blocks in a shuffled pool
    bs = 256
    nb = wd.N_kv // bs
    perm = torch.randperm(wd.B * nb, generator=torch.Generator().manual_seed(wd.seed)).to(dev)

    def paged(t):                                   # [B,H,N,d] -> [B*nb, bs, H, d] in pool order
        blocks = t.view(wd.B, wd.H, nb, bs, wd.d).permute(0, 2, 3, 1, 4).reshape(wd.B * nb, bs, wd.H, wd.d)
        pool = torch.empty_like(blocks)
        pool[perm] = blocks
        return pool
    kc = paged(xd["k"])
    vc = paged(xd["v"])
    qd = xd["q"]
    del xd
    torch.cuda.empty_cache()
    table = perm.view(wd.B, nb).to(torch.int32).contiguous()
    seqlens = torch.full((wd.B,), wd.N_kv, dtype=torch.int32, device=dev)

    def dec_paged(pe):
        if pe is not None:
            pe[0].record(stream)
        fa.fa_decode_paged(qd, kc, vc, od, lsed, table, seqlens, wd.N_kv, wd.scale, wd.n_splits, wsd)
        if pe is not None:
            pe[1].record(stream)
    dp_total, dp_inner = timed(dec_paged, K, inner=True)
    dp_ms = reduce_max(dp_total / K)
    gbs_p = bytes_dec / (statistics.mean(dp_inner) * 1e-3) / 1e9
    breakdown["decode_paged"] = {
        "gbps": round(whole_job_rate(bytes_dec, world, dp_ms * 1e-3) / 1e9, 1),
        "ms": round(dp_ms, 4), "frac_of_hbm": round(gbs_p / peak_hbm, 4),
        "traffic": profiled_traffic("decode_split_kernel<128, paged>", source_digest(
            "exact_io_aware_08_gb300/csrc/decode.cu", "exact_io_aware_08_gb300/csrc/sm103.cuh")),
    }
    clocks = sampler.stop()
    del qd, kc, vc
    torch.cuda.empty_cache()

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": Wm, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{w.name} forward+backward, non-causal (headline)", "B": w.B, "H": w.H,
                   "N": w.N_q, "d": w.d, "causal": False, "scale": "1/sqrt(d)",
                   "step": "fa_fwd + fa_bwd_prep + fa_bwd_main + fa_bwd_finish",
                   "l2": "no flush: each step's inputs (537 MB) exceed the 129 MB L2",
                   "parallelism": f"dp{world} (independent batches per GPU)"},
        "frac_of_peak": round(value / world / peak_tf, 4),
        "breakdown": breakdown,
        "roofline": roofline,
        "e2e": e2e,
        "clocks": clocks,
        "gpu_launches": 4 * K,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = time_oracle(w)
    # last key, so that a reader of the line's tail sees every workload's headline numbers
    result["summary"] = summarize(breakdown, peak_tf)
    return result


def run_reference(args, rank):
    """Reference arm: the fp64 CPU oracle, each step a bounded sample (one whole head)."""
    from exact_io_aware_08_gb300 import inputs
    w = inputs.HEADLINE
    x = head_sample_inputs(w, 1)
    for _ in range(args.warmup):
        oracle_sample_step(x, [(0, 0)], w)
    t0 = time.perf_counter()
    flop = 0
    for _ in range(args.steps):
        flop += oracle_sample_step(x, [(0, 0)], w)
    dt = time.perf_counter() - t0
    value = flop / dt / 1e12
    cores = cpu_cores()
    sample = (f"fp64 NumPy oracle, forward+backward of one whole head of {w.name} per step "
              f"(explicit N x N score matrix); algorithmic FLOP counted")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{w.name} forward+backward, non-causal (headline)", "B": w.B, "H": w.H,
                   "N": w.N_q, "d": w.d, "causal": False},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_profile_case(args):
    """Small single-operation case for ncu captures: warm-up + ``steps`` launches of one op."""
    import torch
    import exact_io_aware_08_gb300 as fa
    from exact_io_aware_08_gb300 import build as fabuild
    from exact_io_aware_08_gb300 import inputs
    fabuild.build()
    fa.load_library()
    B, H, N, d = (int(v) for v in args.shape.split(","))
    scale = d ** -0.5
    if args.profile == "fwd8":
        x = inputs.make_qkv_fp8(B, H, N, N, d, 4242, device="cuda")
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        op = lambda: fa.fa_fwd_fp8(x["q8"], x["k8"], x["v8"], o, lse, scale, x["descale_q"],
                                   x["descale_k"], x["descale_v"], args.causal)
    elif args.profile == "decode_paged":
        x = inputs.make_qkv(B, H, 1, N, d, 4242, with_do=False, device="cuda")
        bs, nb = 256, N // 256
        perm = torch.randperm(B * nb, generator=torch.Generator().manual_seed(7)).cuda()

        def paged(t):
            blocks = t.view(B, H, nb, bs, d).permute(0, 2, 3, 1, 4).reshape(B * nb, bs, H, d)
            pool = torch.empty_like(blocks)
            pool[perm] = blocks
            return pool
        kc, vc = paged(x["k"]), paged(x["v"])
        table = perm.view(B, nb).to(torch.int32).contiguous()
        seqlens = torch.full((B,), N, dtype=torch.int32, device="cuda")
        o = torch.empty_like(x["q"])
        lse = torch.empty((B, H, 1), dtype=torch.float32, device="cuda")
        n_splits = max(1, N // 512)
        ws = torch.empty(fa.fa_decode_workspace_size(B, H, N, d, n_splits), dtype=torch.uint8, device="cuda")
        op = lambda: fa.fa_decode_paged(x["q"], kc, vc, o, lse, table, seqlens, N, scale, n_splits, ws)
    elif args.profile == "decode":
        x = inputs.make_qkv(B, H, 1, N, d, 4242, with_do=False, device="cuda")
        o = torch.empty_like(x["q"])
        lse = torch.empty((B, H, 1), dtype=torch.float32, device="cuda")
        n_splits = max(1, N // 512)
        ws = torch.empty(fa.fa_decode_workspace_size(B, H, N, d, n_splits), dtype=torch.uint8, device="cuda")
        op = lambda: fa.fa_decode_splitkv(x["q"], x["k"], x["v"], o, lse, scale, n_splits, ws)
    else:
        x = {k: v.cuda() for k, v in inputs.make_qkv(B, H, N, N, d, 4242).items()}
        o, lse = fa.forward(x["q"], x["k"], x["v"], causal=args.causal, scale=scale)
        if args.profile == "fwd":
            op = lambda: fa.fa_fwd(x["q"], x["k"], x["v"], o, lse, scale, args.causal)
        else:
            ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, N, d), dtype=torch.uint8, device="cuda")
            dq, dk, dv = (torch.empty_like(x[n]) for n in ("q", "k", "v"))
            op = lambda: fa.fa_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], dq, dk, dv, ws, scale,
                                   args.causal)
    for _ in range(args.warmup + args.steps):
        op()
    fa.fa_sync_status()
    torch.cuda.synchronize()
    print(f"profile case {args.profile} {args.shape} causal={args.causal} done", flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--profile", choices=("fwd", "bwd", "decode", "fwd8", "decode_paged"), default=None,
                    help="run one op on a small case (for ncu) instead of the benchmark")
    ap.add_argument("--shape", default="2,32,4096,128", help="B,H,N,d for --profile")
    ap.add_argument("--causal", action="store_true", help="causal for --profile")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.profile:
        return run_profile_case(args)

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank)), flush=True)
        return 0

    import torch
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", rank=rank, world_size=world)
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
