#!/usr/bin/env python
"""Benchmark: SwiGLU FFN block backward with S3R-EC INT8 on one GB300.

One step = one pass of the whole backward hot path (quantize dY, correction
factors, both INT8 GEMMs of W2, SwiGLU glue fused into the quantization of the
gate/up gradients, their correction factors, both GEMMs of W1 and W3) over one
batch: the d=2048, F=5632, T=8192 (4 x 2048 tokens) Llama-style block, inputs
resident in HBM.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own batch (weak scaling; the path
needs no exchange inside one backward); the time is the max over ranks.
--impl reference times the plain CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import json
import re
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "FFN backward tokens/s, S3R-EC INT8 vs BF16, 1 GB300; quantize GB/s vs HBM peak"
WORKLOAD = "swiglu_ffn_d2048_F5632_T8192"
CFG = workloads.WORKLOADS[WORKLOAD]
T, D, F, S = CFG["T"], CFG["d"], CFG["F"], CFG["S"]
L2_BYTES = 129 * 2 ** 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-context", action="store_true", help="skip the BF16 / baseline-mode context timings")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel-case", choices=["gemm_dx", "gemm_dw", "quantize", "quantize_sweep", "swiglu", "ec", "ffn",
                                              "moe", "fwd", "fwd_gate", "fwd_gate_quantize", "fwd_down",
                                              "sr_bf16", "sr_fp8"],
                    help="profiling helper: run one kernel of the benchmark's block --steps times, print a short line")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (timing only: no collective touches the data path)
# ---------------------------------------------------------------------------
def dist_setup(n):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.idx), "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for nm, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def device_setup(s3r, rank, code_format=None):
    inp = workloads.ffn_inputs(T, D, F, S, seed=workloads.DATA_SEED + 1 + 1000 * rank)
    c = lambda t: t.cuda()
    cf = s3r.DEFAULT_CODES if code_format is None else code_format
    ops = s3r.ffn_forward_operands(c(inp.X), c(inp.W1), c(inp.W3), c(inp.W2), c(inp.a), c(inp.h1), c(inp.h3),
                                   code_format=cf)
    torch.cuda.synchronize()
    return inp, ops


def time_ffn(s3r, ops, dY, steps, warmup, rm, ec, world, events=False):
    """Device time of `steps` ffn_backward calls on resident inputs."""
    ws = torch.empty(s3r.ffn_workspace_size(T, D, F, S, rm, ec, s3r.code_format_of(ops.X8)), dtype=torch.uint8,
                     device="cuda")
    grads = s3r.alloc_ffn_grads(T, D, F)
    st = s3r.new_status()
    for i in range(warmup):
        s3r.ffn_backward(ops, dY, S, rm, ec, seed=i, grads=grads, workspace=ws, status=st)
    step_ev = None
    if events:
        step_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(s3r.FFN_NUM_EVENTS)] for _ in range(steps)]
        for evs in step_ev:
            for e in evs:
                e.record()   # materialize the handles
    torch.cuda.synchronize()
    barrier(world)
    n0 = s3r.kernel_launch_count()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(steps):
        s3r.ffn_backward(ops, dY, S, rm, ec, seed=1000 + i, grads=grads, workspace=ws, status=st,
                         step_events=step_ev[i] if events else None)
    t1.record()
    torch.cuda.synchronize()
    launches = s3r.kernel_launch_count() - n0
    ms = t0.elapsed_time(t1)
    barrier(world)
    s3r.check_status(st)
    seg = None
    if events:
        seg = np.array([[evs[j].elapsed_time(evs[j + 1]) for j in range(s3r.FFN_NUM_EVENTS - 1)] for evs in step_ev])
    return max_over_ranks(ms, world), launches, seg, grads


def time_e2e(s3r, inp, ops, steps, warmup, world):
    """Same step through the C ABI with HOST buffers: pinned host -> device
    copies of every input of the step, the backward, device -> host copies of
    all four gradients, inside the timed region."""
    host_in = {k: getattr(ops, k).cpu().pin_memory() for k in
               ("X8", "s_x", "A8", "s_a", "W1_8", "s_w1", "W3_8", "s_w3", "W2_8", "s_w2", "h1", "h3")}
    host_in["dY"] = inp.dY.pin_memory()
    dev_in = {k: torch.empty_like(v, device="cuda") for k, v in host_in.items()}
    dops = s3r.FFNOperands(**{k: dev_in[k] for k in host_in if k != "dY"})
    grads = s3r.alloc_ffn_grads(T, D, F)
    host_out = {k: torch.empty(getattr(grads, k).shape, dtype=torch.float32).pin_memory()
                for k in ("dX", "dW1", "dW3", "dW2")}
    ws = torch.empty(s3r.ffn_workspace_size(T, D, F, S, code_format=s3r.code_format_of(ops.X8)), dtype=torch.uint8,
                     device="cuda")
    bi = sum(v.numel() * v.element_size() for v in host_in.values())
    bo = sum(v.numel() * v.element_size() for v in host_out.values())

    def step(i):
        for k, v in host_in.items():
            dev_in[k].copy_(v, non_blocking=True)
        s3r.ffn_backward(dops, dev_in["dY"], S, seed=i, grads=grads, workspace=ws)
        for k, v in host_out.items():
            v.copy_(getattr(grads, k), non_blocking=True)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    barrier(world)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(steps):
        step(i)
    t1.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1), world)
    barrier(world)
    return ms, bi, bo


def time_bf16_backward(inp, steps, warmup):
    """Context: the same block's backward in BF16 with cuBLAS via torch."""
    X, W1, W3, W2, h1, h3, a, dY = (t.cuda() for t in (inp.X, inp.W1, inp.W3, inp.W2, inp.h1, inp.h3, inp.a, inp.dY))

    def step():
        dA = dY @ W2.t()
        dW2 = a.t() @ dY
        s = torch.sigmoid(h1.float())
        dAf = dA.float()
        dh1 = (dAf * h3.float() * s * (1 + h1.float() * (1 - s))).to(torch.bfloat16)
        dh3 = (dAf * h1.float() * s).to(torch.bfloat16)
        dX = dh1 @ W1.t() + dh3 @ W3.t()
        dW1 = X.t() @ dh1
        dW3 = X.t() @ dh3
        return dX, dW1, dW2, dW3

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        step()
    t1.record()
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps


def time_moe(s3r, steps=5, warmup=2):
    """Context: the mixture-of-experts workload (8 experts, d=4096, F=1408,
    16384 tokens top-2, Zipf(1.1) loads): grouped S3R-EC two-way backward
    through ffn_backward, and the same per-expert backward in BF16 with cuBLAS."""
    w = workloads.WORKLOADS["moe_e8_d4096_F1408_tok16384_top2"]
    inp = workloads.moe_inputs(w["tokens"], w["topk"], w["experts"], w["d"], w["F"], seed=workloads.DATA_SEED + 5)
    c = lambda t: t.cuda()
    ops = s3r.moe_forward_operands(c(inp.X), c(inp.W1), c(inp.W3), c(inp.W2), c(inp.a), c(inp.h1), c(inp.h3))
    dY = inp.dY.cuda()
    offs = inp.offsets
    st = s3r.new_status()
    grads = s3r.ffn_backward(ops, dY, 0, group_offsets=offs, status=st)
    ws = torch.empty(s3r.grouped_workspace_size(offs, w["d"], w["F"]), dtype=torch.uint8, device="cuda")

    def ours():
        s3r.ffn_backward(ops, dY, 0, grads=grads, workspace=ws, status=st, group_offsets=offs)

    X, W1, W3, W2, h1, h3, a = (c(t) for t in (inp.X, inp.W1, inp.W3, inp.W2, inp.h1, inp.h3, inp.a))

    def bf16():
        for e in range(w["experts"]):
            r0, r1 = offs[e], offs[e + 1]
            g, x, hh1, hh3, aa = dY[r0:r1], X[r0:r1], h1[r0:r1], h3[r0:r1], a[r0:r1]
            dA = g @ W2[e].t()
            aa.t() @ g
            s = torch.sigmoid(hh1.float())
            dAf = dA.float()
            dh1 = (dAf * hh3.float() * s * (1 + hh1.float() * (1 - s))).to(torch.bfloat16)
            dh3 = (dAf * hh1.float() * s).to(torch.bfloat16)
            dh1 @ W1[e].t() + dh3 @ W3[e].t()
            x.t() @ dh1
            x.t() @ dh3

    out = {}
    # per-step split of one grouped call (each step over all experts)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(s3r.FFN_NUM_EVENTS)]
    for e_ in ev:
        e_.record()
    torch.cuda.synchronize()
    s3r.ffn_backward(ops, dY, 0, grads=grads, workspace=ws, status=st, group_offsets=offs, step_events=ev)
    torch.cuda.synchronize()
    out["step_breakdown_ms"] = {n: round(ev[j].elapsed_time(ev[j + 1]), 4) for j, n in enumerate(s3r.FFN_STEPS)}
    for name, fn in (("s3r_ec_two_way_grouped", ours), ("bf16_cublas_per_expert", bf16)):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(steps):
            fn()
        t1.record()
        torch.cuda.synchronize()
        ms = t0.elapsed_time(t1) / steps
        out[name] = {"tokens_s": round(w["tokens"] / (ms * 1e-3), 1), "ms": round(ms, 4)}
    s3r.check_status(st)
    out["group_rows"] = [b - a for a, b in zip(offs[:-1], offs[1:])]
    out["speedup_vs_bf16"] = round(out["bf16_cublas_per_expert"]["ms"] / out["s3r_ec_two_way_grouped"]["ms"], 3)
    return out


def time_ffn_large(s3r, steps=5, warmup=2):
    """Context: the larger SwiGLU block (d=4096, F=14336, T=16384 = 8 x 2048,
    Table III's W7 shape): S3R-EC two-way, S3R-EC dX-only, S3R, independent SR
    and the BF16 cuBLAS backward of the same block."""
    w = workloads.WORKLOADS["swiglu_ffn_d4096_F14336_T16384"]
    Tl, dl, Fl, Sl = w["T"], w["d"], w["F"], w["S"]
    inp = workloads.ffn_inputs(Tl, dl, Fl, Sl, seed=workloads.DATA_SEED + 2)
    c = lambda t: t.cuda()
    ops = s3r.ffn_forward_operands(c(inp.X), c(inp.W1), c(inp.W3), c(inp.W2), c(inp.a), c(inp.h1), c(inp.h3))
    dY = inp.dY.cuda()
    st = s3r.new_status()
    out = {}
    for name, rm, ec in (("s3r_ec_two_way", s3r.ROUND_S3R, s3r.EC_TWO_WAY), ("s3r_ec_dx_only", s3r.ROUND_S3R,
                         s3r.EC_DX_ONLY), ("s3r", s3r.ROUND_S3R, s3r.EC_NONE), ("indep_sr_int8", s3r.ROUND_INDEP,
                         s3r.EC_NONE)):
        ws = torch.empty(s3r.ffn_workspace_size(Tl, dl, Fl, Sl, rm, ec), dtype=torch.uint8, device="cuda")
        grads = s3r.alloc_ffn_grads(Tl, dl, Fl)
        for i in range(warmup):
            s3r.ffn_backward(ops, dY, Sl, rm, ec, seed=i, grads=grads, workspace=ws, status=st)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for i in range(steps):
            s3r.ffn_backward(ops, dY, Sl, rm, ec, seed=100 + i, grads=grads, workspace=ws, status=st)
        t1.record()
        torch.cuda.synchronize()
        ms = t0.elapsed_time(t1) / steps
        out[name] = {"tokens_s": round(Tl / (ms * 1e-3), 1), "ms": round(ms, 4),
                     "gemm_tflops_if_all_gemm": round(12.0 * Tl * dl * Fl / (ms * 1e-3) / 1e12, 1)}
        del ws, grads
    s3r.check_status(st)
    bms = time_bf16_backward(inp, steps, warmup)
    out["bf16_cublas_backward"] = {"tokens_s": round(Tl / (bms * 1e-3), 1), "ms": round(bms, 4)}
    out["s3r_ec_two_way_vs_bf16"] = round(bms / out["s3r_ec_two_way"]["ms"], 3)
    out["s3r_ec_two_way_vs_indep_sr"] = round(out["indep_sr_int8"]["ms"] / out["s3r_ec_two_way"]["ms"], 3)
    return out


def _event_ms(fn, steps, warmup):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        fn()
    t1.record()
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps


def time_forward(s3r, inp, pk, steps=10, warmup=3):
    """Context: the block's INT8 forward (ffn_forward: RTNE X and weights, the
    gate/up GEMM with the SwiGLU gate in its epilogue, RTNE a, the down GEMM),
    its two GEMMs alone, and the BF16 cuBLAS forward of the same block."""
    c = lambda t: t.cuda()
    X, W1, W3, W2 = c(inp.X), c(inp.W1), c(inp.W3), c(inp.W2)
    st = s3r.new_status()
    out = s3r.alloc_ffn_forward(T, D, F, keep_a=False)   # the backward reads a's codes only
    fwd = lambda: s3r.ffn_forward(X, W1, W3, W2, out=out, status=st)
    ms = _event_ms(fwd, steps, warmup)
    o = out.ops
    gate = lambda: s3r.int8_gemm_fwd_swiglu(o.X8, o.s_x, o.W1_8, o.s_w1, o.W3_8, o.s_w3, o.h1, o.h3,
                                            with_gate=False, status=st)
    gms = _event_ms(gate, steps, warmup)
    gq = lambda: s3r.swiglu_fwd_quantize(o.h1, o.h3, keep_a=False, Q=o.A8, scale=o.s_a, status=st)
    qms = _event_ms(gq, steps, warmup)
    down = lambda: s3r.int8_gemm_fwd(o.A8, o.s_a, o.W2_8, o.s_w2, Y=out.Y, status=st)
    dms = _event_ms(down, steps, warmup)
    s3r.check_status(st)

    def bf16():
        h1, h3 = X @ W1, X @ W3
        a = (torch.nn.functional.silu(h1.float()) * h3.float()).to(torch.bfloat16)
        return a @ W2

    bms = _event_ms(bf16, steps, warmup)
    peak = pk.get("bf16_tflops")
    tf = lambda flops, t: round(flops / (t * 1e-3) / 1e12, 1)
    return {"ms": round(ms, 4), "tokens_s": round(T / (ms * 1e-3), 1), "tflops": tf(6.0 * T * D * F, ms),
            "gate_up_gemm": {"ms": round(gms, 4), "tflops": tf(4.0 * T * D * F, gms),
                             "frac_bf16_burst": round(4.0 * T * D * F / (gms * 1e-3) / 1e12 / peak, 3)},
            "swiglu_gate_rtne_a": {"ms": round(qms, 4),
                                   "GB_s": round(6.0 * T * F / (qms * 1e-3) / 1e9, 1),
                                   "frac_hbm": round(6.0 * T * F / (qms * 1e-3) / 1e9 / pk["hbm_gbs"], 3)},
            "down_gemm": {"ms": round(dms, 4), "tflops": tf(2.0 * T * D * F, dms),
                          "frac_bf16_burst": round(2.0 * T * D * F / (dms * 1e-3) / 1e12 / peak, 3)},
            "bf16_cublas_forward": {"ms": round(bms, 4), "tokens_s": round(T / (bms * 1e-3), 1)},
            "vs_bf16": round(bms / ms, 3)}


def time_sr_bf16(s3r, pk, steps=20, warmup=3):
    """Context: stochastic rounding of fp32 to bf16 on the hardware conversion
    with S3R's per-token thresholds, per-element thresholds, and RTNE, at
    [16384, 8192] (fp32 in, bf16 out: 6 algorithmic bytes per element; 805 MB
    per call, larger than L2)."""
    Tq, Nq = 16384, 8192
    G = (workloads.quantize_sweep_input(Tq, Nq, seed=workloads.DATA_SEED + 3).float() * 1e3).cuda()
    Y = torch.empty((Tq, Nq), dtype=torch.bfloat16, device="cuda")
    out = {"shape": [Tq, Nq]}
    for name, rm in (("s3r", s3r.ROUND_S3R), ("indep_sr", s3r.ROUND_INDEP), ("rtne", s3r.ROUND_RTNE)):
        ms = _event_ms(lambda: s3r.s3r_sr_bf16(G, rm, seed=1, Y=Y), steps, warmup)
        gbs = 6.0 * Tq * Nq / (ms * 1e-3) / 1e9
        out[name] = {"us": round(ms * 1e3, 2), "GB_s": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 3)}
    # the same rounding to FP8 e4m3 after a scale (fp32 in, one byte out: 5 B per element)
    Y8 = torch.empty((Tq, Nq), dtype=torch.uint8, device="cuda")
    for name, rm in (("fp8_s3r", s3r.ROUND_S3R), ("fp8_indep_sr", s3r.ROUND_INDEP), ("fp8_rtne", s3r.ROUND_RTNE)):
        ms = _event_ms(lambda: s3r.s3r_sr_fp8(G, 0.01, rm, seed=1, Y=Y8), steps, warmup)
        gbs = 5.0 * Tq * Nq / (ms * 1e-3) / 1e9
        out[name] = {"us": round(ms * 1e3, 2), "GB_s": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 3)}
    del G, Y, Y8
    return out


def time_quantize_sweep(s3r, steps=20):
    """S3R / independent SR / RTNE quantizers on dY [16384, 8192] bf16 with 1% x100
    outliers; int8 codes (1 B) and fp16-carried codes (2 B)."""
    Tq, Nq = 16384, 8192
    G = workloads.quantize_sweep_input(Tq, Nq, seed=workloads.DATA_SEED + 3).cuda()
    out = {}
    S8, F16 = s3r.CODES_S8, s3r.CODES_F16
    q8 = s3r.s3r_quantize(G, code_format=S8)
    q16 = s3r.s3r_quantize(G, code_format=F16)
    qi = s3r.indep_sr_quantize(G, code_format=S8)
    Qr, sr = s3r.rtne_quantize(G, code_format=S8)
    part = 8 / 128   # the two fp32 error partials per 128 elements
    runs = {
        "s3r": (lambda i: s3r.s3r_quantize(G, seed=i, out=q8), 2 + 1 + part),
        "s3r_f16_codes": (lambda i: s3r.s3r_quantize(G, seed=i, out=q16), 2 + 2 + part),
        "indep_sr_one_copy": (lambda i: s3r.indep_sr_quantize(G, seed=i, out=qi), 3.0),
        "rtne": (lambda i: s3r.rtne_quantize(G, Q=Qr, scale=sr), 3.0),
        # the paper's thresholds (7-bit, four per word) and its per-tensor step (one extra read
        # of the gradient for the global absmax before the quantization pass)
        "s3r_7bit": (lambda i: s3r.s3r_quantize_ex(G, round_mode=s3r.ROUND_S3R_7BIT, seed=i, out=q8), 2 + 1 + part),
        "s3r_7bit_per_tensor": (lambda i: s3r.s3r_quantize_ex(G, round_mode=s3r.ROUND_S3R_7BIT, per_tensor=True,
                                                              seed=i, out=q8), 2 + 2 + 1 + part),
    }
    for name, (fn, bpe) in runs.items():
        for i in range(3):
            fn(i)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for i in range(steps):
            fn(i)
        t1.record()
        torch.cuda.synchronize()
        ms = t0.elapsed_time(t1) / steps
        out[name] = {"us": round(ms * 1e3, 2), "GB_s": round(bpe * Tq * Nq / (ms * 1e-3) / 1e9, 1),
                     "alg_bytes_per_elem": round(bpe, 4)}
    out["shape"] = [Tq, Nq]
    # the other row counts of the sweep, S3R with int8 codes
    for Tx in (4096, 65536):
        Gx = workloads.quantize_sweep_input(Tx, Nq, seed=workloads.DATA_SEED + 3).cuda()
        qx = s3r.s3r_quantize(Gx, code_format=S8)
        for i in range(3):
            s3r.s3r_quantize(Gx, seed=i, out=qx)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for i in range(steps):
            s3r.s3r_quantize(Gx, seed=i, out=qx)
        t1.record()
        torch.cuda.synchronize()
        ms = t0.elapsed_time(t1) / steps
        out[f"s3r_T{Tx}"] = {"us": round(ms * 1e3, 2), "GB_s": round((3 + part) * Tx * Nq / (ms * 1e-3) / 1e9, 1),
                             "alg_bytes_per_elem": round(3 + part, 4),
                             "l2_note": "input 64 MB < L2: repeated calls partly hit L2" if Tx == 4096 else ""}
        del Gx, qx
    return out


def cpu_baseline(tokens=128):
    """The plain CPU oracle (single thread) on a bounded sample of the same
    block: `tokens` tokens (one example) of the d=2048, F=5632 FFN."""
    import oracle as orc
    inp = workloads.ffn_inputs(tokens, D, F, tokens, seed=workloads.DATA_SEED + 1)
    f = orc.from_torch_bf16
    ops = orc.ffn_forward_operands(f(inp.X), f(inp.W1), f(inp.W3), f(inp.W2), f(inp.a))
    h1, h3, dY = f(inp.h1), f(inp.h3), f(inp.dY)
    t0 = time.perf_counter()
    orc.ffn_backward(ops, h1, h3, dY, tokens, mode=orc.S3R, ec_mode=orc.EC_TWO_WAY, seed=0)
    dt = time.perf_counter() - t0
    return {"value": round(tokens / dt, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{tokens} tokens (one example) of the d=2048, F=5632 SwiGLU block, S3R-EC two-way, "
                      f"{dt:.1f} s single-threaded"}


def profiled_traffic(kernel: str):
    """DRAM bytes per GEMM product of `kernel` from the committed ncu summary
    of this workload, or None when the GEMM source changed since the capture."""
    import hashlib
    root = os.path.dirname(os.path.abspath(__file__))
    try:
        txt = open(os.path.join(root, "profiles", "ffn_d2048_F5632_T8192_launches.md")).read()
        src = open(os.path.join(root, "stochastic_rounding_int8_gb300", "csrc", "gemm_umma.cu"), "rb").read()
    except OSError:
        return None
    m = re.search(r"gemm_umma\.cu sha256: ([0-9a-f]{64})", txt)
    t = re.search(rf"{re.escape(kernel)}=(\d+)", txt)
    if not m or not t or m.group(1) != hashlib.sha256(src).hexdigest():
        return None
    return int(t.group(1))


def run_ours(args, world, rank, local):
    import stochastic_rounding_int8_gb300 as s3r
    s3r.lib()
    pk, pk_kind = peaks()
    inp, ops = device_setup(s3r, rank)
    dY = inp.dY.cuda()
    clocks = Clocks(local)
    # main timed region: S3R-EC two-way, step events for the per-kernel roofline
    clocks.start()
    ms, launches, seg, _ = time_ffn(s3r, ops, dY, args.steps, args.warmup, s3r.ROUND_S3R, s3r.EC_TWO_WAY, world,
                                    events=True)
    clk = clocks.stop()
    ms_step = ms / args.steps
    value = world * T * args.steps / (ms * 1e-3)
    # per-step segments -> dominant kernel class
    segm = seg.mean(0)
    names = s3r.FFN_STEPS
    # second field: GEMM products of 2*T*d*F flops per step; with fp16 codes dA + dW2 and
    # dX1 + dX3 + dW1 + dW3 are one mixed launch each, so all six products form one class
    classes = {"int8_gemm": (segm[2] + segm[3] + segm[6] + segm[7], 6),
               "quantize (dY + SwiGLU-fused)": (segm[0] + segm[4], 2), "s3r_ec_correct": (segm[1] + segm[5], 3)}
    dom = max(classes, key=lambda k: classes[k][0])
    dom_ms, dom_n = classes[dom]
    flops_per_launch = 2.0 * T * D * F
    if dom.startswith("int8_gemm"):
        achieved = flops_per_launch / (dom_ms / dom_n * 1e-3) / 1e12
        peak = pk.get("bf16_tflops_sustained", pk.get("bf16_tflops"))
        roof = {"kernel": "umma_gemm_kernel (int8_gemm_dx / int8_gemm_dw: dA + dW2 and dX1 + dX3 + dW1 + dW3 "
                          "as two mixed launches)", "bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": profiled_traffic(dom),
                "traffic_note": "DRAM read + write bytes per GEMM product from the committed ncu capture "
                                "(profiles/ffn_d2048_F5632_T8192_launches.md); null once the GEMM source changed",
                "peak_note": f"dense bf16 sustained ({pk_kind}); the s8 codes run on the tensor cores at the "
                             f"16-bit rate or below on sm_103a",
                "flops_per_product": flops_per_launch, "products_per_step": dom_n,
                "avg_us_per_product": round(dom_ms / dom_n * 1e3, 1)}
    else:
        roof = {"kernel": dom, "bound": "hbm", "achieved": None, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": None, "traffic": None}
    steps_ms = {n: round(float(v), 4) for n, v in zip(names, segm)}
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "s8", "data": "synthetic (seeded; shapes/distributions of the paper's FFN "
                                                  "block workload)",
        "config": {"workload": WORKLOAD, "T": T, "d": D, "F": F, "examples": T // S, "seq": S,
                   "rounding": "S3R Phi_2D", "ec": "two-way", "tile": 128,
                   "codes": "int8 values carried in fp16 (tcgen05 kind::f16, fp32 accumulate per 128-K block)",
                   "l2": "working set ~1 GB > 129 MB L2 (no flush needed)", "parallelism": f"replica x{world}"},
        "clocks": clk,
        "gpu_launches": int(launches),
        "roofline": roof,
        "step_breakdown_ms": steps_ms,
    }
    # e2e through the C ABI with host buffers
    e2e_steps = max(3, min(args.steps, 20))
    ems, bi, bo = time_e2e(s3r, inp, ops, e2e_steps, min(args.warmup, 3), world)
    line["e2e"] = {"value": round(world * T * e2e_steps / (ems * 1e-3), 1), "unit": "tokens/s",
                   "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": e2e_steps}
    if not args.no_context and rank == 0:
        ctx = {}
        for name, rm, ec in (("s3r_ec_dx_only", s3r.ROUND_S3R, s3r.EC_DX_ONLY), ("s3r", s3r.ROUND_S3R, s3r.EC_NONE),
                             ("indep_sr_int8", s3r.ROUND_INDEP, s3r.EC_NONE), ("rtne_int8", s3r.ROUND_RTNE, s3r.EC_NONE),
                             # the paper's own variants: 7-bit thresholds, Phi_bcast, the dW-only correction
                             ("s3r_7bit_ec_two_way", s3r.ROUND_S3R_7BIT, s3r.EC_TWO_WAY),
                             ("s3r_bcast_ec_two_way", s3r.ROUND_BCAST, s3r.EC_TWO_WAY),
                             ("s3r_ec_dw_only", s3r.ROUND_S3R, s3r.EC_DW_ONLY)):
            m, _, _, _ = time_ffn(s3r, ops, dY, 10, 2, rm, ec, 1)
            ctx[name] = {"tokens_s": round(T * 10 / (m * 1e-3), 1), "ms": round(m / 10, 4)}
        _, ops8 = device_setup(s3r, rank, s3r.CODES_S8)
        m, _, _, _ = time_ffn(s3r, ops8, dY, 5, 1, s3r.ROUND_S3R, s3r.EC_TWO_WAY, 1)
        ctx["s3r_ec_two_way_int8_storage_mma_sync"] = {"tokens_s": round(T * 5 / (m * 1e-3), 1), "ms": round(m / 5, 4)}
        del ops8
        bms = time_bf16_backward(inp, 10, 3)
        ctx["bf16_cublas_backward"] = {"tokens_s": round(T / (bms * 1e-3), 1), "ms": round(bms, 4)}
        ctx["s3r_ec_two_way_vs_bf16"] = round(ctx["bf16_cublas_backward"]["ms"] / ms_step, 3)
        ctx["s3r_ec_two_way_vs_indep_sr"] = round(ctx["indep_sr_int8"]["ms"] / ms_step, 3)
        fw = time_forward(s3r, inp, pk)
        ctx["forward_int8"] = fw
        # one INT8 training step of the block: this forward + the timed backward
        ctx["train_step_int8_vs_bf16"] = {
            "int8_ms": round(fw["ms"] + ms_step, 4),
            "bf16_ms": round(fw["bf16_cublas_forward"]["ms"] + ctx["bf16_cublas_backward"]["ms"], 4)}
        qs = time_quantize_sweep(s3r)
        for k in ("s3r", "s3r_f16_codes", "indep_sr_one_copy", "rtne", "s3r_7bit", "s3r_7bit_per_tensor",
                  "s3r_T4096", "s3r_T65536"):
            qs[k]["frac_hbm"] = round(qs[k]["GB_s"] / pk["hbm_gbs"], 3)
        ctx["quantize_sweep"] = qs
        ctx["sr_bf16_sweep"] = time_sr_bf16(s3r, pk)
        ctx["moe_e8_d4096_F1408_tok16384_top2"] = time_moe(s3r)
        ctx["swiglu_ffn_d4096_F14336_T16384"] = time_ffn_large(s3r)
        line["context"] = ctx
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    return line


def run_kernel_case(args):
    """Launch one kernel class of the benchmark's FFN block (the W2 / W1 linear
    shapes) --steps times after --warmup, for ncu captures; prints its time."""
    import stochastic_rounding_int8_gb300 as s3r
    s3r.lib()
    inp, ops = device_setup(s3r, 0)
    dY = inp.dY.cuda()
    q2 = s3r.s3r_quantize(dY, ops.s_a, ops.s_w2)
    ec2 = s3r.s3r_ec_correct(q2, T, D, S, ops.W2_8, ops.A8, s3r.EC_TWO_WAY)
    dA = s3r.int8_gemm_dx(q2.Q, q2.tile_scale, ops.W2_8, ops.s_a, s3r.EC_TWO_WAY, ec2, S)
    fns = {
        "gemm_dx": lambda: s3r.int8_gemm_dx(q2.Q, q2.tile_scale, ops.W2_8, ops.s_a, s3r.EC_TWO_WAY, ec2, S, dX=dA),
        "gemm_dw": lambda: s3r.int8_gemm_dw(ops.A8, q2.Q, q2.tile_scale, ops.s_w2, s3r.EC_TWO_WAY, ec2, S),
        "quantize": lambda: s3r.s3r_quantize(dY, ops.s_a, ops.s_w2, out=q2),
        "swiglu": lambda: s3r.swiglu_quantize(dA, ops.h1, ops.h3, ops.s_x, ops.s_w1, ops.s_w3),
        "ec": lambda: s3r.s3r_ec_correct(q2, T, D, S, ops.W2_8, ops.A8, s3r.EC_TWO_WAY),
        "ffn": lambda: s3r.ffn_backward(ops, dY, S),
    }
    if args.kernel_case == "moe":
        w = workloads.WORKLOADS["moe_e8_d4096_F1408_tok16384_top2"]
        mi = workloads.moe_inputs(w["tokens"], w["topk"], w["experts"], w["d"], w["F"], seed=workloads.DATA_SEED + 5)
        c = lambda t: t.cuda()
        mops = s3r.moe_forward_operands(c(mi.X), c(mi.W1), c(mi.W3), c(mi.W2), c(mi.a), c(mi.h1), c(mi.h3))
        mdY = mi.dY.cuda()
        fns["moe"] = lambda: s3r.ffn_backward(mops, mdY, 0, group_offsets=mi.offsets)
    if args.kernel_case.startswith("fwd"):
        c = lambda t: t.cuda()
        X, W1, W3, W2 = c(inp.X), c(inp.W1), c(inp.W3), c(inp.W2)
        fo = s3r.ffn_forward(X, W1, W3, W2, keep_a=False)
        o = fo.ops
        fns["fwd"] = lambda: s3r.ffn_forward(X, W1, W3, W2, out=fo)
        fns["fwd_gate"] = lambda: s3r.int8_gemm_fwd_swiglu(o.X8, o.s_x, o.W1_8, o.s_w1, o.W3_8, o.s_w3, o.h1, o.h3,
                                                           with_gate=False)
        fns["fwd_gate_quantize"] = lambda: s3r.swiglu_fwd_quantize(o.h1, o.h3, keep_a=False, Q=o.A8, scale=o.s_a)
        fns["fwd_down"] = lambda: s3r.int8_gemm_fwd(o.A8, o.s_a, o.W2_8, o.s_w2, Y=fo.Y)
    if args.kernel_case in ("sr_bf16", "sr_fp8"):
        Gb = (workloads.quantize_sweep_input(16384, 8192, seed=workloads.DATA_SEED + 3).float() * 1e3).cuda()
        Yb = torch.empty((16384, 8192), dtype=torch.bfloat16, device="cuda")
        fns["sr_bf16"] = lambda: s3r.s3r_sr_bf16(Gb, s3r.ROUND_S3R, seed=1, Y=Yb)
        Y8b = torch.empty((16384, 8192), dtype=torch.uint8, device="cuda")
        fns["sr_fp8"] = lambda: s3r.s3r_sr_fp8(Gb, 0.01, s3r.ROUND_S3R, seed=1, Y=Y8b)
    if args.kernel_case == "quantize_sweep":
        Gs = workloads.quantize_sweep_input(16384, 8192, seed=workloads.DATA_SEED + 3).cuda()
        qs = s3r.s3r_quantize(Gs, code_format=s3r.CODES_S8)
        fns["quantize_sweep"] = lambda: s3r.s3r_quantize(Gs, out=qs)
    fn = fns[args.kernel_case]
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        fn()
    t1.record()
    torch.cuda.synchronize()
    print(json.dumps({"kernel_case": args.kernel_case, "ms_per_call": round(t0.elapsed_time(t1) / args.steps, 4)}))


def run_reference(args, world, rank):
    """The oracle as the reference arm: each step a bounded sample (8 tokens of
    the d=2048, F=5632 block, ~1-3 s) on the host cores."""
    if rank != 0:
        return None
    import oracle as orc
    tok = 8
    inp = workloads.ffn_inputs(tok, D, F, tok, seed=workloads.DATA_SEED + 1)
    f = orc.from_torch_bf16
    ops = orc.ffn_forward_operands(f(inp.X), f(inp.W1), f(inp.W3), f(inp.W2), f(inp.a))
    h1, h3, dY = f(inp.h1), f(inp.h3), f(inp.dY)
    run = lambda: orc.ffn_backward(ops, h1, h3, dY, tok, mode=orc.S3R, ec_mode=orc.EC_TWO_WAY, seed=0)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    value = tok * args.steps / dt
    sample = f"{tok} tokens (one example) of the d=2048, F=5632 SwiGLU block per step, single-threaded C oracle"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "s8", "data": "synthetic",
            "config": {"workload": WORKLOAD, "T": T, "d": D, "F": F, "rounding": "S3R Phi_2D", "ec": "two-way"},
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    world, rank, local = dist_setup(args.gpus)
    if args.kernel_case:
        run_kernel_case(args)
        return
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    else:
        line = run_ours(args, world, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
