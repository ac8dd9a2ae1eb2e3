"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This module only draws random tensors with the shapes and distributions of the
S3R paper's workloads ("Efficient Quantization Training with Stochastic
Rounding via Structured Subspace Randomness", §IV-A and Table III). It holds
none of the method's arithmetic: no scaling, rounding, thresholds or error
correction. The paper's own workloads (C4 text, MaxText models) are not
available; these draws stand in for them through their shapes only.

Distributions:
  * activations X ~ N(0, 1), weights W ~ N(0, 0.02^2) (std 0.02);
  * upstream gradient dY = 1e-3 * Student-t(df=3);
  * SwiGLU pre-activations h1, h3 ~ N(0, (0.02*sqrt(d))^2), the marginal law of
    X @ W for the X, W above, drawn directly instead of multiplying;
  * quantize sweep: dY as above with 1% of elements (i.i.d. Bernoulli(0.01))
    multiplied by 100;
  * MoE: expert row counts proportional to (e+1)^-1.1 (Zipf, s = 1.1), rounded
    by largest remainder to the routed row total.

Everything is returned as torch CPU tensors (bf16 where the layer stores bf16);
callers copy them to the device themselves.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

# Data seed convention: 1234 + workload index.
DATA_SEED = 1234


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _bf16(a: np.ndarray) -> torch.Tensor:
    """float32/64 numpy array -> contiguous torch.bfloat16 (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def normal_bf16(rng: np.random.Generator, shape, std: float) -> torch.Tensor:
    return _bf16(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


def student_t_bf16(rng: np.random.Generator, shape, scale: float = 1e-3, df: float = 3.0,
                   outlier_frac: float = 0.0, outlier_mult: float = 100.0) -> torch.Tensor:
    t = rng.standard_t(df, size=shape).astype(np.float32) * np.float32(scale)
    if outlier_frac > 0.0:
        mask = rng.random(shape, dtype=np.float32) < np.float32(outlier_frac)
        t = np.where(mask, t * np.float32(outlier_mult), t)
    return _bf16(t)


@dataclass
class LinearInputs:
    X: torch.Tensor      # bf16 [T, K]
    W: torch.Tensor      # bf16 [K, N]
    dY: torch.Tensor     # bf16 [T, N]
    S: int               # tokens per example (T = B*S)


def linear_inputs(T: int, K: int, N: int, S: int | None = None, seed: int = DATA_SEED) -> LinearInputs:
    """One linear layer Y = X W and its upstream gradient (tiny-linear workload)."""
    rng = _rng(seed)
    X = normal_bf16(rng, (T, K), 1.0)
    W = normal_bf16(rng, (K, N), 0.02)
    dY = student_t_bf16(rng, (T, N))
    return LinearInputs(X, W, dY, T if S is None else S)


@dataclass
class FFNInputs:
    X: torch.Tensor      # bf16 [T, d]
    W1: torch.Tensor     # bf16 [d, F]  (gate)
    W3: torch.Tensor     # bf16 [d, F]  (up)
    W2: torch.Tensor     # bf16 [F, d]  (down)
    h1: torch.Tensor     # bf16 [T, F]  saved gate pre-activation
    h3: torch.Tensor     # bf16 [T, F]  saved up pre-activation
    a: torch.Tensor      # bf16 [T, F]  saved input of W2: silu(h1) * h3 (forward pass)
    dY: torch.Tensor     # bf16 [T, d]
    S: int


def ffn_inputs(T: int, d: int, F: int, S: int, seed: int = DATA_SEED) -> FFNInputs:
    """A Llama-style SwiGLU FFN block's saved forward state and upstream gradient."""
    rng = _rng(seed)
    X = normal_bf16(rng, (T, d), 1.0)
    W1 = normal_bf16(rng, (d, F), 0.02)
    W3 = normal_bf16(rng, (d, F), 0.02)
    W2 = normal_bf16(rng, (F, d), 0.02)
    std_h = 0.02 * math.sqrt(d)
    h1 = normal_bf16(rng, (T, F), std_h)
    h3 = normal_bf16(rng, (T, F), std_h)
    # Forward activation of the block (not part of the backward method).
    a = (torch.nn.functional.silu(h1.float()) * h3.float()).to(torch.bfloat16)
    dY = student_t_bf16(rng, (T, d))
    return FFNInputs(X, W1, W3, W2, h1, h3, a, dY, S)


def quantize_sweep_input(T: int, N: int, seed: int = DATA_SEED) -> torch.Tensor:
    """Heavy-tailed gradient with 1% x100 outliers (quantize-only sweep)."""
    return student_t_bf16(_rng(seed), (T, N), outlier_frac=0.01)


def moe_group_sizes(rows: int, experts: int, s: float = 1.1) -> list[int]:
    """Zipf(s) expert loads, normalised and rounded by largest remainder."""
    w = np.array([(e + 1) ** (-s) for e in range(experts)], dtype=np.float64)
    exact = rows * w / w.sum()
    base = np.floor(exact).astype(np.int64)
    rem = rows - int(base.sum())
    order = np.argsort(-(exact - base), kind="stable")
    base[order[:rem]] += 1
    return [int(x) for x in base]


@dataclass
class MoEInputs:
    X: torch.Tensor      # bf16 [R, d]   expert-sorted routed rows
    W1: torch.Tensor     # bf16 [E, d, F]
    W3: torch.Tensor     # bf16 [E, d, F]
    W2: torch.Tensor     # bf16 [E, F, d]
    h1: torch.Tensor     # bf16 [R, F]
    h3: torch.Tensor     # bf16 [R, F]
    a: torch.Tensor      # bf16 [R, F]
    dY: torch.Tensor     # bf16 [R, d]
    offsets: list[int]   # [E+1] row offsets of each expert's group


def moe_inputs(tokens: int, topk: int, experts: int, d: int, F: int, seed: int = DATA_SEED) -> MoEInputs:
    return moe_inputs_sized(moe_group_sizes(tokens * topk, experts), d, F, seed)


def moe_inputs_sized(sizes, d: int, F: int, seed: int = DATA_SEED) -> MoEInputs:
    """Routed rows for explicit per-expert group sizes (expert-sorted)."""
    rng = _rng(seed)
    experts = len(sizes)
    offsets = [0]
    for n in sizes:
        offsets.append(offsets[-1] + n)
    R = offsets[-1]
    X = normal_bf16(rng, (R, d), 1.0)
    W1 = normal_bf16(rng, (experts, d, F), 0.02)
    W3 = normal_bf16(rng, (experts, d, F), 0.02)
    W2 = normal_bf16(rng, (experts, F, d), 0.02)
    std_h = 0.02 * math.sqrt(d)
    h1 = normal_bf16(rng, (R, F), std_h)
    h3 = normal_bf16(rng, (R, F), std_h)
    a = (torch.nn.functional.silu(h1.float()) * h3.float()).to(torch.bfloat16)
    dY = student_t_bf16(rng, (R, d))
    return MoEInputs(X, W1, W3, W2, h1, h3, a, dY, offsets)


# The five synthetic workloads, by what they are.
WORKLOADS = {
    "tiny_linear_T256_K512_N1024": dict(kind="linear", T=256, K=512, N=1024, S=256),
    "swiglu_ffn_d2048_F5632_T8192": dict(kind="ffn", T=8192, d=2048, F=5632, S=2048),
    "swiglu_ffn_d4096_F14336_T16384": dict(kind="ffn", T=16384, d=4096, F=14336, S=2048),
    "quantize_sweep_N8192": dict(kind="quantize", N=8192, Ts=(4096, 16384, 65536)),
    "moe_e8_d4096_F1408_tok16384_top2": dict(kind="moe", tokens=16384, topk=2, experts=8, d=4096, F=1408),
}
