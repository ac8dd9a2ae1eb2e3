"""Pins for the oracle's SwiGLU backward glue (the FFN block of the S3R paper,
§IV-A / Table III): its exp against the C library's exp, its sigmoid against
the fp64 definition, and the gate/up gradients against torch autograd (a
library routine) in fp64."""
import math

import numpy as np
import torch


def _ulp32(x):
    x = np.float32(abs(x))
    return float(np.spacing(x)) if x > 0 else float(np.spacing(np.float32(0)))


def test_expf_within_two_ulp(orc):
    xs = np.linspace(-87.0, 88.0, 60001, dtype=np.float32)
    xs = np.concatenate([xs, np.float32([0.0, -0.0, 1e-8, -1e-8, 0.5, -0.5, 1.0, 10.0, -10.0])])
    worst = 0.0
    for x in xs:
        got = orc.expf(float(x))
        ref = math.exp(float(np.float32(x)))
        worst = max(worst, abs(got - ref) / _ulp32(ref))
    assert worst <= 2.0, worst


def test_expf_clamps_to_normal_range(orc):
    assert orc.expf(200.0) == orc.expf(88.0) and math.isfinite(orc.expf(200.0))
    assert orc.expf(-200.0) == orc.expf(-87.0) > 0.0


def test_sigmoid_close_to_definition(orc):
    worst = 0.0
    for x in np.linspace(-30, 30, 20001, dtype=np.float32):
        ref = 1.0 / (1.0 + math.exp(-float(x)))
        worst = max(worst, abs(orc.sigmoidf(float(x)) - ref) / _ulp32(ref))
    assert worst <= 4.0, worst
    assert orc.sigmoidf(0.0) == 0.5


def test_swiglu_grads_match_autograd(orc):
    rng = np.random.default_rng(0)
    n = 50000
    h1 = (rng.standard_normal(n) * 2).astype(np.float32)
    h3 = (rng.standard_normal(n) * 2).astype(np.float32)
    dA = rng.standard_normal(n).astype(np.float32)
    dh1, dh3 = orc.swiglu_bwd(dA, h1, h3)
    t1 = torch.tensor(h1, dtype=torch.float64, requires_grad=True)
    t3 = torch.tensor(h3, dtype=torch.float64, requires_grad=True)
    a = torch.nn.functional.silu(t1) * t3
    a.backward(torch.tensor(dA, dtype=torch.float64))
    g1, g3 = t1.grad.numpy(), t3.grad.numpy()
    scale1 = np.abs(dA * h3).astype(np.float64) + 1e-30
    scale3 = np.abs(dA * h1).astype(np.float64) + 1e-30
    assert np.max(np.abs(dh1 - g1) / scale1) < 2e-6
    assert np.max(np.abs(dh3 - g3) / scale3) < 2e-6
