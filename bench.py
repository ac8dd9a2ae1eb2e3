#!/usr/bin/env python
"""Benchmark: SwiGLU FFN block backward with S3R-EC INT8 on one GB300.

One step = one pass of the whole backward hot path (quantize dY, correction
factors, both INT8 GEMMs of W2, SwiGLU glue fused into the quantization of the
gate/up gradients, their correction factors, both GEMMs of W1 and W3) over one
batch: the d=4096, F=14336, T=16384 (8 x 2048 tokens) Llama-style block (the
shape of the paper's Table III row W7, the largest FFN block of the workloads),
inputs resident in HBM.  The d=2048, F=5632, T=8192 block and the other
workloads are timed as context.  Prints ONE JSON line (rank 0).

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
WORKLOAD = "swiglu_ffn_d4096_F14336_T16384"
SMALL_BLOCK = "swiglu_ffn_d2048_F5632_T8192"
CFG = workloads.WORKLOADS[WORKLOAD]
T, D, F, S = CFG["T"], CFG["d"], CFG["F"], CFG["S"]
L2_BYTES = 129 * 2 ** 20
E2E_IN_STREAMS = 3   # streams carrying the e2e input copies (one stream: 0.55 M tokens/s on one box, 1.33 M with 2-4)

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the two GEMM launches of one
# ffn_backward step, divided by the step's six products, from a one-pass ncu capture of
#   python bench.py --kernel-case ffn --block <block> --steps 1 --warmup 1
# on a GB300; keyed by the sha256 of the GEMM sources it was taken on (the kernel, then the tile
# deal), so that it is reported only while they are unchanged, then by block.
GEMM_TRAFFIC = {
    "8e8c1dafe7b0a96ca2b0f918c7f71b02e0250f042eb21bfbbf09ccee94839d98": {
        "swiglu_ffn_d4096_F14336_T16384": 2237.7e6,   # dA + dW2 4398 MB, dX1 + dX3 + dW1 + dW3 9028 MB
        "swiglu_ffn_d2048_F5632_T8192": 209.5e6,      # 441.5 MB and 815.4 MB
    },
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-context", action="store_true", help="skip the BF16 / baseline-mode context timings")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel-case", choices=["gemm_dx", "gemm_dw", "quantize", "quantize_sweep", "swiglu", "ec", "ffn",
                                              "moe", "fwd", "fwd_gate", "fwd_gate_quantize", "fwd_down",
                                              "sr_bf16", "sr_fp8"],
                    help="profiling helper: run one kernel of a block --steps times, print a short line")
    ap.add_argument("--block", choices=[WORKLOAD, SMALL_BLOCK], default=SMALL_BLOCK,
                    help="--kernel-case: which FFN block (default: the smaller one, for ncu captures)")
    ap.add_argument("--fuse-glue", action="store_true",
                    help="--kernel-case ffn: the SwiGLU glue inside the dA GEMM's epilogue (S3R_FFN_FUSE_GLUE)")
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
class Block:
    """One SwiGLU FFN block workload: its sizes and its seeded inputs."""

    def __init__(self, name, data_seed):
        w = workloads.WORKLOADS[name]
        self.name = name
        self.T, self.d, self.F, self.S = w["T"], w["d"], w["F"], w["S"]
        self.data_seed = data_seed
        self.flops_per_product = 2.0 * self.T * self.d * self.F   # each of the six GEMM products of a step
        # algorithmic bytes of the six products (each reads its two code operands once and writes its
        # fp32 output once; dX1 and dX3 share one dX), averaged per product
        T, d, F = self.T, self.d, self.F
        step = ((2 * T * d + 2 * F * d + 4 * T * F) + (2 * T * F + 2 * T * d + 4 * F * d)
                + 2 * (2 * T * F + 2 * F * d) + 4 * T * d + 2 * (2 * T * d + 2 * T * F + 4 * d * F))
        self.gemm_bytes_per_product = step / 6.0

    def inputs(self, rank=0):
        return workloads.ffn_inputs(self.T, self.d, self.F, self.S, seed=self.data_seed + 1000 * rank)


HEAD = Block(WORKLOAD, workloads.DATA_SEED + 2)
SMALL = Block(SMALL_BLOCK, workloads.DATA_SEED + 1)


def device_ops(s3r, inp, code_format=None):
    c = lambda t: t.cuda()
    cf = s3r.DEFAULT_CODES if code_format is None else code_format
    ops = s3r.ffn_forward_operands(c(inp.X), c(inp.W1), c(inp.W3), c(inp.W2), c(inp.a), c(inp.h1), c(inp.h3),
                                   code_format=cf)
    torch.cuda.synchronize()
    return ops


def time_ffn(s3r, blk, ops, dY, steps, warmup, rm, ec, world, events=False, fuse=False, widen=False):
    """Device time of `steps` ffn_backward calls on resident inputs: total ms
    between two events around the loop, launches counted by the library, and
    (events=True) each step's per-step-boundary event times [steps, 8].
    fuse: the SwiGLU glue inside the dA GEMM's epilogue.  widen: int8 operand
    codes widened inside the call (S3R_CODES_S8_F16)."""
    T, d, F, S = blk.T, blk.d, blk.F, blk.S
    fmt = s3r.CODES_S8_F16 if widen else s3r.code_format_of(ops.X8)
    ws = torch.empty(s3r.ffn_workspace_size(T, d, F, S, rm, ec, fmt), dtype=torch.uint8, device="cuda")
    grads = s3r.alloc_ffn_grads(T, d, F)
    st = s3r.new_status()
    for i in range(warmup):
        s3r.ffn_backward(ops, dY, S, rm, ec, seed=i, grads=grads, workspace=ws, status=st, fuse_glue=fuse,
                         widen_codes=widen)
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
                         step_events=step_ev[i] if events else None, fuse_glue=fuse, widen_codes=widen)
    t1.record()
    torch.cuda.synchronize()
    launches = s3r.kernel_launch_count() - n0
    ms = t0.elapsed_time(t1)
    barrier(world)
    s3r.check_status(st)
    seg = None
    if events:
        seg = np.array([[evs[j].elapsed_time(evs[j + 1]) for j in range(s3r.FFN_NUM_EVENTS - 1)] for evs in step_ev])
    del ws, grads
    return max_over_ranks(ms, world), launches, seg


E2E_CODES = ("X8", "A8", "W1_8", "W3_8", "W2_8")


def time_e2e(s3r, blk, inp, ops, steps, warmup, world, int8_at_rest=True, recompute_a=True):
    """Same step through the C ABI with HOST buffers: every step copies all of
    its inputs from pinned host memory to the device, runs the backward, and
    copies all four gradients back, inside the timed region.  The copies run
    on their own streams, double-buffered, so step i's input copy and step
    i - 1's gradient copy overlap step i - 1's and step i's backward (the
    way a training loop feeds a device); events order the buffers' reuse.
    int8_at_rest: the operand codes live in host memory as int8 (half the
    bytes over the host link) and the call widens them on the device
    (S3R_CODES_S8_F16); otherwise they are copied as fp16 codes.  recompute_a:
    the codes of a and their scales are not kept by the forward; the call forms
    them from h1 and h3 (S3R_FFN_RECOMPUTE_A)."""
    T, d, F, S = blk.T, blk.d, blk.F, blk.S
    conv = (lambda k, t: t.to(torch.int8) if k in E2E_CODES else t) if int8_at_rest else (lambda k, t: t)
    keys = ("X8", "s_x", "A8", "s_a", "W1_8", "s_w1", "W3_8", "s_w3", "W2_8", "s_w2", "h1", "h3")
    host_in = {k: conv(k, getattr(ops, k)).cpu().pin_memory() for k in keys
               if not (recompute_a and k in ("A8", "s_a"))}
    host_in["dY"] = inp.dY.pin_memory()
    dev_in = [{k: torch.empty_like(v, device="cuda") for k, v in host_in.items()} for _ in range(2)]
    dops = [s3r.FFNOperands(**{k: di.get(k) for k in keys}) for di in dev_in]
    grads = [s3r.alloc_ffn_grads(T, d, F) for _ in range(2)]
    host_out = [{k: torch.empty(getattr(grads[0], k).shape, dtype=torch.float32).pin_memory()
                 for k in ("dX", "dW1", "dW3", "dW2")} for _ in range(2)]
    fmt = s3r.CODES_S8_F16 if int8_at_rest else s3r.code_format_of(ops.X8)
    flags = s3r.FFN_RECOMPUTE_A if recompute_a else 0
    ws = torch.empty(s3r.ffn_workspace_size(T, d, F, S, code_format=fmt, flags=flags), dtype=torch.uint8,
                     device="cuda")
    bi = sum(v.numel() * v.element_size() for v in host_in.values())
    bo = sum(v.numel() * v.element_size() for v in host_out[0].values())
    # the input copies spread over N_IN streams (balanced by bytes), so several copy engines share them
    N_IN = E2E_IN_STREAMS
    s_ins = [torch.cuda.Stream() for _ in range(N_IN)]
    s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    load = [0] * N_IN
    lane_of = {}
    for k, v in sorted(host_in.items(), key=lambda kv: -kv[1].numel() * kv[1].element_size()):
        j = load.index(min(load))
        lane_of[k] = j
        load[j] += v.numel() * v.element_size()
    ev = lambda: torch.cuda.Event()
    in_done = [[ev() for _ in range(N_IN)] for _ in range(2)]
    comp_done, out_done = [ev(), ev()], [ev(), ev()]
    used = [False, False]

    def step(i):
        b = i % 2
        for j, s_in in enumerate(s_ins):
            with torch.cuda.stream(s_in):
                if used[b]:
                    s_in.wait_event(comp_done[b])    # the backward of step i - 2 has read these inputs
                for k, v in host_in.items():
                    if lane_of[k] == j:
                        dev_in[b][k].copy_(v, non_blocking=True)
                in_done[b][j].record(s_in)
        with torch.cuda.stream(s_comp):
            for j in range(N_IN):
                s_comp.wait_event(in_done[b][j])
            if used[b]:
                s_comp.wait_event(out_done[b])   # step i - 2's gradients have left the device
            s3r.ffn_backward(dops[b], dev_in[b]["dY"], S, seed=i, grads=grads[b], workspace=ws, stream=s_comp,
                             widen_codes=int8_at_rest, recompute_a=recompute_a)
            comp_done[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            for k, v in host_out[b].items():
                v.copy_(getattr(grads[b], k), non_blocking=True)
            out_done[b].record(s_out)
        used[b] = True

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    barrier(world)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_ins[0])
    for s_in in s_ins[1:]:
        s_in.wait_event(t0)
    for i in range(steps):
        step(warmup + i)
    s_out.wait_event(out_done[(warmup + steps - 1) % 2])
    s_out.wait_event(comp_done[(warmup + steps - 1) % 2])
    t1.record(s_out)
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1), world)
    barrier(world)
    del dev_in, dops, grads, ws, host_in, host_out
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

    return _event_ms(step, steps, warmup)


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


def gemm_roofline(blk, seg, pk, pk_kind):
    """The GEMM class of ffn_backward (dA + dW2 and dX1 + dX3 + dW1 + dW3, two
    mixed tcgen05 launches carrying the six products of a step) from the step
    events: algorithmic flops per product over the class's mean time per
    product, against the measured dense bf16 peak (burst: the GEMMs are timed
    in a step-long region at full clock, not in a seconds-long loop)."""
    segm = seg.mean(0)
    gemm_ms = float(segm[2] + segm[3] + segm[6] + segm[7])
    achieved = blk.flops_per_product / (gemm_ms / 6 * 1e-3) / 1e12
    peak = pk["bf16_tflops"]
    return {"kernel": "umma_gemm_kernel (dA + dW2 and dX1 + dX3 + dW1 + dW3 as two mixed launches)",
            "bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4),
            "peak_note": f"dense bf16 burst ({pk_kind}); the codes run on the tensor cores as fp16 (kind::f16, "
                         f"the same nominal rate as bf16)",
            "frac_of_sustained_peak": round(achieved / pk.get("bf16_tflops_sustained", peak), 4),
            "flops_per_product": blk.flops_per_product, "products_per_step": 6,
            "avg_us_per_product": round(gemm_ms / 6 * 1e3, 1)}


def gemm_traffic(blk):
    """DRAM bytes per GEMM product of block `blk` from the recorded ncu capture,
    or None when the GEMM source changed since it was taken."""
    import hashlib
    csrc = os.path.join(ROOT, "stochastic_rounding_int8_gb300", "csrc")
    h = hashlib.sha256()
    try:
        for f in ("gemm_umma.cu", "deal_plan.h"):   # the kernel and the tile deal it walks
            h.update(open(os.path.join(csrc, f), "rb").read())
    except OSError:
        return None
    return GEMM_TRAFFIC.get(h.hexdigest(), {}).get(blk.name)


def add_traffic(roof, blk):
    """The GEMM class's recorded DRAM traffic per product next to its algorithmic bytes."""
    tr = gemm_traffic(blk)
    roof["traffic"] = tr
    roof["algorithmic_bytes_per_product"] = round(blk.gemm_bytes_per_product)
    roof["traffic_over_algorithmic"] = round(tr / blk.gemm_bytes_per_product, 3) if tr else None
    roof["traffic_note"] = ("DRAM read + write bytes per GEMM product of this block from a one-pass ncu capture of "
                            "the step's two GEMM launches; null when the GEMM source changed since")


def block_line(s3r, blk, inp, ops, dY, steps, warmup, world, pk, pk_kind):
    """Timed S3R-EC two-way steps of one block: throughput, mean and median step
    time, the step split and the GEMM class's roofline."""
    ms, launches, seg = time_ffn(s3r, blk, ops, dY, steps, warmup, s3r.ROUND_S3R, s3r.EC_TWO_WAY, world,
                                 events=True)
    per_step = seg.sum(1)
    return {"tokens_s": world * blk.T * steps / (ms * 1e-3), "ms_per_step": ms / steps,
            "ms_per_step_median": float(np.median(per_step)), "launches": launches,
            "step_breakdown_ms": {n: round(float(v), 4) for n, v in zip(s3r.FFN_STEPS, seg.mean(0))},
            "roofline": gemm_roofline(blk, seg, pk, pk_kind)}


def mode_context(s3r, blk, ops, dY, inp, steps=8, warmup=2):
    """The same block under the other rounding / correction modes, int8 code
    storage (the mma.sync path, and widened to fp16 inside the call) and the
    BF16 cuBLAS backward."""
    ctx = {}
    for name, rm, ec in (("s3r_ec_dx_only", s3r.ROUND_S3R, s3r.EC_DX_ONLY), ("s3r", s3r.ROUND_S3R, s3r.EC_NONE),
                         ("indep_sr_int8", s3r.ROUND_INDEP, s3r.EC_NONE), ("rtne_int8", s3r.ROUND_RTNE, s3r.EC_NONE),
                         # the paper's own variants: 7-bit thresholds, Phi_bcast, the dW-only correction
                         ("s3r_7bit_ec_two_way", s3r.ROUND_S3R_7BIT, s3r.EC_TWO_WAY),
                         ("s3r_bcast_ec_two_way", s3r.ROUND_BCAST, s3r.EC_TWO_WAY),
                         ("s3r_ec_dw_only", s3r.ROUND_S3R, s3r.EC_DW_ONLY)):
        m, _, _ = time_ffn(s3r, blk, ops, dY, steps, warmup, rm, ec, 1)
        ctx[name] = {"tokens_s": round(blk.T * steps / (m * 1e-3), 1), "ms": round(m / steps, 4)}
    # the SwiGLU glue inside the dA GEMM's epilogue (S3R_FFN_FUSE_GLUE) against the separate kernel
    m, _, seg = time_ffn(s3r, blk, ops, dY, steps, warmup, s3r.ROUND_S3R, s3r.EC_TWO_WAY, 1, events=True, fuse=True)
    ctx["s3r_ec_two_way_fused_glue"] = {"tokens_s": round(blk.T * steps / (m * 1e-3), 1), "ms": round(m / steps, 4),
                                        "dA_dW2_launch_ms": round(float(seg[:, 2].mean()), 4)}
    ops8 = device_ops(s3r, inp, s3r.CODES_S8)
    m, _, _ = time_ffn(s3r, blk, ops8, dY, 3, 1, s3r.ROUND_S3R, s3r.EC_TWO_WAY, 1)
    ctx["s3r_ec_two_way_int8_storage_mma_sync"] = {"tokens_s": round(blk.T * 3 / (m * 1e-3), 1), "ms": round(m / 3, 4)}
    # the same int8 operand codes widened to fp16 inside the call, then the tcgen05 block
    m, _, _ = time_ffn(s3r, blk, ops8, dY, steps, warmup, s3r.ROUND_S3R, s3r.EC_TWO_WAY, 1, widen=True)
    ctx["s3r_ec_two_way_int8_codes_widened"] = {"tokens_s": round(blk.T * steps / (m * 1e-3), 1),
                                                "ms": round(m / steps, 4)}
    del ops8
    bms = time_bf16_backward(inp, steps, warmup)
    ctx["bf16_cublas_backward"] = {"tokens_s": round(blk.T / (bms * 1e-3), 1), "ms": round(bms, 4)}
    return ctx


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
        ms = _event_ms(fn, steps, warmup)
        out[name] = {"tokens_s": round(w["tokens"] / (ms * 1e-3), 1), "ms": round(ms, 4)}
    s3r.check_status(st)
    out["group_rows"] = [b - a for a, b in zip(offs[:-1], offs[1:])]
    out["speedup_vs_bf16"] = round(out["bf16_cublas_per_expert"]["ms"] / out["s3r_ec_two_way_grouped"]["ms"], 3)
    return out


def time_forward(s3r, blk, inp, pk, steps=10, warmup=3):
    """Context: the block's INT8 forward (ffn_forward: RTNE X and weights, the
    gate/up GEMM, the SwiGLU gate fused into the RTNE of a, the down GEMM),
    its two GEMMs and the gate kernel alone, and the BF16 cuBLAS forward of the
    same block."""
    T, D, F = blk.T, blk.d, blk.F
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
    peak = pk["bf16_tflops"]
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


def time_quantize_sweep(s3r, pk, steps=20):
    """S3R / independent SR / RTNE quantizers on dY [T, 8192] bf16 with 1% x100
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
        it = iter(range(10 ** 9))
        ms = _event_ms(lambda: fn(next(it)), steps, 3)
        gbs = bpe * Tq * Nq / (ms * 1e-3) / 1e9
        out[name] = {"us": round(ms * 1e3, 2), "GB_s": round(gbs, 1), "alg_bytes_per_elem": round(bpe, 4),
                     "frac_hbm": round(gbs / pk["hbm_gbs"], 3)}
    out["shape"] = [Tq, Nq]
    # the other row counts of the sweep, S3R with int8 codes
    for Tx in (4096, 65536):
        Gx = workloads.quantize_sweep_input(Tx, Nq, seed=workloads.DATA_SEED + 3).cuda()
        qx = s3r.s3r_quantize(Gx, code_format=S8)
        it = iter(range(10 ** 9))
        ms = _event_ms(lambda: s3r.s3r_quantize(Gx, seed=next(it), out=qx), steps, 3)
        gbs = (3 + part) * Tx * Nq / (ms * 1e-3) / 1e9
        out[f"s3r_T{Tx}"] = {"us": round(ms * 1e3, 2), "GB_s": round(gbs, 1), "alg_bytes_per_elem": round(3 + part, 4),
                             "frac_hbm": round(gbs / pk["hbm_gbs"], 3),
                             "l2_note": "input 64 MB < L2: repeated calls partly hit L2" if Tx == 4096 else ""}
        del Gx, qx
    return out


def host_cpu():
    """The host's logical core count and CPU model (lscpu, else /proc/cpuinfo)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        m = re.search(r"^Model name:\s*(.+)$", out, re.M)
        model = m.group(1).strip() if m else None
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            m = re.search(r"^model name\s*:\s*(.+)$", open("/proc/cpuinfo").read(), re.M)
            model = m.group(1).strip() if m else None
        except OSError:
            pass
    return {"host_cores": os.cpu_count(), "cpu_model": model or "unknown"}


def _oracle_block_sample(blk, tokens):
    """The oracle's operands for `tokens` tokens (one example) of a block."""
    import oracle as orc
    inp = workloads.ffn_inputs(tokens, blk.d, blk.F, tokens, seed=blk.data_seed)
    f = orc.from_torch_bf16
    ops = orc.ffn_forward_operands(f(inp.X), f(inp.W1), f(inp.W3), f(inp.W2), f(inp.a))
    h1, h3, dY = f(inp.h1), f(inp.h3), f(inp.dY)
    return lambda: orc.ffn_backward(ops, h1, h3, dY, tokens, mode=orc.S3R, ec_mode=orc.EC_TWO_WAY, seed=0)


def cpu_baseline(blk, tokens=64):
    """The plain CPU oracle (single thread, as it stands) on a bounded sample of
    the timed block: `tokens` tokens (one example) of its backward."""
    run = _oracle_block_sample(blk, tokens)
    t0 = time.perf_counter()
    run()
    dt = time.perf_counter() - t0
    return {"value": round(tokens / dt, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{tokens} tokens (one example) of the d={blk.d}, F={blk.F} SwiGLU block backward, S3R-EC "
                      f"two-way, {dt:.1f} s on one thread of the host", **host_cpu()}


def config_of(blk, world):
    return {"workload": blk.name, "T": blk.T, "d": blk.d, "F": blk.F, "examples": blk.T // blk.S, "seq": blk.S,
            "rounding": "S3R Phi_2D", "ec": "two-way", "tile": 128,
            "codes": "int8 values carried in fp16 (tcgen05 kind::f16, fp32 accumulate per 128-K block)",
            "l2": "working set of a step several GB > 129 MB L2 (no flush needed)", "parallelism": f"replica x{world}"}


def run_ours(args, world, rank, local):
    import stochastic_rounding_int8_gb300 as s3r
    s3r.lib()
    pk, pk_kind = peaks()
    blk = HEAD
    inp = blk.inputs(rank)
    ops = device_ops(s3r, inp)
    dY = inp.dY.cuda()
    clocks = Clocks(local)
    # main timed region: S3R-EC two-way, step events for the per-kernel roofline
    clocks.start()
    r = block_line(s3r, blk, inp, ops, dY, args.steps, args.warmup, world, pk, pk_kind)
    clk = clocks.stop()
    roof = r["roofline"]
    add_traffic(roof, blk)
    line = {
        "metric": METRIC, "value": round(r["tokens_s"], 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(r["ms_per_step"], 4),
        "ms_per_step_median": round(r["ms_per_step_median"], 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "s8", "data": "synthetic (seeded; shapes/distributions of the paper's FFN "
                                                    "block workload)",
        "config": config_of(blk, world),
        "clocks": clk,
        "gpu_launches": int(r["launches"]),
        "roofline": roof,
        "step_breakdown_ms": r["step_breakdown_ms"],
    }
    # e2e through the C ABI with host buffers
    # as many steps as the device-timed leg: the timed region includes filling the copy pipeline
    # (the first step's inputs) and draining it (the last step's gradients)
    e2e_steps = max(3, args.steps)
    # the host link is shared with the machine's other work and its rate swings between runs:
    # three runs, the median reported, all three listed
    runs = []
    for _ in range(3):
        ems, bi, bo = time_e2e(s3r, blk, inp, ops, e2e_steps, min(args.warmup, 2), world)
        runs.append(world * blk.T * e2e_steps / (ems * 1e-3))
    line["e2e"] = {"value": round(sorted(runs)[1], 1), "unit": "tokens/s",
                   "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": e2e_steps,
                   "runs": [round(v, 1) for v in runs], "statistic": "median of the runs",
                   "copies": "every step copies all inputs in and all four gradients out; the copies run on their "
                             "own streams, double-buffered, overlapping the neighbouring steps' backward",
                   "operand_codes_at_rest": "int8 (ffn_backward widens them on the device, S3R_CODES_S8_F16)",
                   "codes_of_a": "formed by the call from h1 and h3 (S3R_FFN_RECOMPUTE_A), not copied"}
    if not args.no_context and rank == 0:
        ctx = mode_context(s3r, blk, ops, dY, inp)
        ctx["s3r_ec_two_way_vs_bf16"] = round(ctx["bf16_cublas_backward"]["ms"] / r["ms_per_step"], 3)
        ems16, bi16, bo16 = time_e2e(s3r, blk, inp, ops, e2e_steps, min(args.warmup, 2), world, int8_at_rest=False,
                                     recompute_a=False)
        ctx["e2e_fp16_codes_at_rest"] = {"tokens_s": round(world * blk.T * e2e_steps / (ems16 * 1e-3), 1),
                                         "h2d_bytes_per_step": bi16, "d2h_bytes_per_step": bo16}
        ctx["s3r_ec_two_way_vs_indep_sr"] = round(ctx["indep_sr_int8"]["ms"] / r["ms_per_step"], 3)
        # what keeping the activation gradient dA in fp32 costs: written by the dA GEMM, read by the
        # SwiGLU quantizer (the fused-glue variant above avoids it but stalls the GEMM instead)
        da_bytes = 2 * 4 * blk.T * blk.F
        ctx["dA_fp32_intermediate"] = {"bytes_per_step": da_bytes,
                                       "ms_at_measured_hbm": round(da_bytes / (pk["hbm_gbs"] * 1e9) * 1e3, 4)}
        fw = time_forward(s3r, blk, inp, pk)
        ctx["forward_int8"] = fw
        # one INT8 training step of the block: this forward + the timed backward
        ctx["train_step_int8_vs_bf16"] = {
            "int8_ms": round(fw["ms"] + r["ms_per_step"], 4),
            "bf16_ms": round(fw["bf16_cublas_forward"]["ms"] + ctx["bf16_cublas_backward"]["ms"], 4)}
        del ops, dY, inp
        torch.cuda.empty_cache()
        # the smaller block as its own line
        sb = SMALL
        sinp = sb.inputs()
        sops = device_ops(s3r, sinp)
        sdY = sinp.dY.cuda()
        rs = block_line(s3r, sb, sinp, sops, sdY, 20, 3, 1, pk, pk_kind)
        add_traffic(rs["roofline"], sb)
        sctx = {"tokens_s": round(rs["tokens_s"], 1), "ms_per_step": round(rs["ms_per_step"], 4),
                "ms_per_step_median": round(rs["ms_per_step_median"], 4),
                "step_breakdown_ms": rs["step_breakdown_ms"], "roofline": rs["roofline"]}
        sctx.update(mode_context(s3r, sb, sops, sdY, sinp))
        sctx["s3r_ec_two_way_vs_bf16"] = round(sctx["bf16_cublas_backward"]["ms"] / rs["ms_per_step"], 3)
        sctx["s3r_ec_two_way_vs_indep_sr"] = round(sctx["indep_sr_int8"]["ms"] / rs["ms_per_step"], 3)
        sctx["forward_int8"] = time_forward(s3r, sb, sinp, pk)
        ctx[sb.name] = sctx
        del sops, sdY, sinp
        torch.cuda.empty_cache()
        ctx["quantize_sweep"] = time_quantize_sweep(s3r, pk)
        ctx["sr_bf16_sweep"] = time_sr_bf16(s3r, pk)
        ctx["moe_e8_d4096_F1408_tok16384_top2"] = time_moe(s3r)
        line["context"] = ctx
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(blk)
    return line


def run_kernel_case(args):
    """Launch one kernel class of an FFN block (its W2 / W1 linear shapes)
    --steps times after --warmup, for ncu captures; prints its time."""
    import stochastic_rounding_int8_gb300 as s3r
    s3r.lib()
    blk = HEAD if args.block == WORKLOAD else SMALL
    T, D, F, S = blk.T, blk.d, blk.F, blk.S
    inp = blk.inputs()
    ops = device_ops(s3r, inp)
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
    }
    if args.kernel_case == "ffn":
        ws = torch.empty(s3r.ffn_workspace_size(T, D, F, S), dtype=torch.uint8, device="cuda")
        grads = s3r.alloc_ffn_grads(T, D, F)
        fns["ffn"] = lambda: s3r.ffn_backward(ops, dY, S, grads=grads, workspace=ws, fuse_glue=args.fuse_glue)
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
    ms = _event_ms(fns[args.kernel_case], args.steps, args.warmup)
    print(json.dumps({"kernel_case": args.kernel_case, "block": blk.name, "ms_per_call": round(ms, 4)}))


def run_reference(args, world, rank):
    """The oracle as the reference arm: each step a bounded sample (4 tokens of
    the timed block, one example; a few seconds) on one host thread."""
    if rank != 0:
        return None
    blk = HEAD
    tok = 4
    run = _oracle_block_sample(blk, tok)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    value = tok * args.steps / dt
    sample = (f"{tok} tokens (one example) of the d={blk.d}, F={blk.F} SwiGLU block backward per step, "
              f"single-threaded C oracle")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "s8", "data": "synthetic",
            "config": config_of(blk, world),
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": sample, **host_cpu()},
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
