"""Pin for the oracle's composition of the SwiGLU FFN block backward.

The INT8 backward estimates the backward pass of the executed forward graph
through the dequantized operands ([S3R] §III-A, §III-C "First-order
unbiasedness": "every layer's gradient is unbiased with respect to the
backward pass of the executed forward graph (with X_hat, W_hat if it is
quantized)").  So the oracle's chained outputs must sit within quantization
noise of torch autograd in fp64 through diag(s_x) X_hat, W_hat diag(s_w); a
mis-wired step (swapped operand, transposition, scale) lands far outside.
"""
import numpy as np
import pytest
import torch

import workloads


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.fixture(scope="module")
def small_ffn(orc):
    inp = workloads.ffn_inputs(T=256, d=128, F=384, S=128, seed=5)
    X, W1, W3, W2 = (orc.from_torch_bf16(t) for t in (inp.X, inp.W1, inp.W3, inp.W2))
    h1, h3, a, dY = (orc.from_torch_bf16(t) for t in (inp.h1, inp.h3, inp.a, inp.dY))
    ops = orc.ffn_forward_operands(X, W1, W3, W2, a)
    return inp, ops, h1, h3, dY


def _autograd_ref(ops, h1, h3, dY):
    f = lambda q, s, ax: torch.tensor(q, dtype=torch.float64) * torch.tensor(s, dtype=torch.float64).unsqueeze(1 - ax)
    Xd = f(ops.X8, ops.s_x, 0)
    Ad = f(ops.A8, ops.s_a, 0)
    W1d, W3d, W2d = f(ops.W1_8, ops.s_w1, 1), f(ops.W3_8, ops.s_w3, 1), f(ops.W2_8, ops.s_w2, 1)
    G = torch.tensor(dY, dtype=torch.float64)
    dW2 = Ad.T @ G
    dA = G @ W2d.T
    t1 = torch.tensor(h1, dtype=torch.float64, requires_grad=True)
    t3 = torch.tensor(h3, dtype=torch.float64, requires_grad=True)
    (torch.nn.functional.silu(t1) * t3).backward(dA)
    dh1, dh3 = t1.grad, t3.grad
    return dict(dW2=dW2.numpy(), dA=dA.numpy(), dX=(dh1 @ W1d.T + dh3 @ W3d.T).numpy(),
                dW1=(Xd.T @ dh1).numpy(), dW3=(Xd.T @ dh3).numpy())


@pytest.mark.parametrize("mode,ec", [("S3R", "EC_TWO_WAY"), ("S3R", "EC_DX_ONLY"), ("S3R", "EC_NONE"),
                                     ("INDEP", "EC_NONE"), ("RTNE", "EC_NONE")])
def test_ffn_chain_within_quantization_noise(orc, small_ffn, mode, ec):
    _, ops, h1, h3, dY = small_ffn
    ref = _autograd_ref(ops, h1, h3, dY)
    out = orc.ffn_backward(ops, h1, h3, dY, 128, mode=getattr(orc, mode), ec_mode=getattr(orc, ec), seed=1)
    errs = dict(dA=_rel(out.dA, ref["dA"]), dW2=_rel(out.dW2, ref["dW2"]), dX=_rel(out.dX, ref["dX"]),
                dW1=_rel(out.dW1, ref["dW1"]), dW3=_rel(out.dW3, ref["dW3"]))
    for k, e in errs.items():
        assert e < 0.15, (k, errs)
    # a mis-wired glue (gate and up gradients swapped) is far outside that band
    assert _rel(out.dW1, ref["dW3"]) > 0.5


def test_ffn_first_stage_unbiased(orc, small_ffn):
    """Averaging the W2 stage over seeds converges to the exact product."""
    _, ops, h1, h3, dY = small_ffn
    ref = _autograd_ref(ops, h1, h3, dY)
    n = 64
    acc = None
    for s in range(n):
        lb = orc.linear_backward(dY, ops.A8, ops.s_a, ops.W2_8, ops.s_w2, 128, mode=orc.S3R,
                                 ec_mode=orc.EC_TWO_WAY, seed=s, tensor_id=orc.TID_W2)
        acc = lb.dX if acc is None else acc + lb.dX
    one = orc.linear_backward(dY, ops.A8, ops.s_a, ops.W2_8, ops.s_w2, 128, mode=orc.S3R,
                              ec_mode=orc.EC_TWO_WAY, seed=0, tensor_id=orc.TID_W2).dX
    e1, en = _rel(one, ref["dA"]), _rel(acc / n, ref["dA"])
    assert en < e1 / 4, (e1, en)      # ~ 1/sqrt(64) = 1/8 of the single-seed error
