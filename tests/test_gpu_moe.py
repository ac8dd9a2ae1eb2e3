"""GPU parity: the grouped (mixture-of-experts) SwiGLU backward.

1. ffn_backward in grouped mode equals, bit for bit, the block backward run
   by separate library calls on each expert's rows with tensor ids 16 e +
   (0, 1, 2); empty experts get zero weight gradients.
2. Each expert's staged backward matches the oracle's grouped backward (the
   same near-tie rules as the dense block).
The MoE workload at full size is compared with the oracle, expert by expert,
in test_gpu_ffn_oracle.py.
"""
import numpy as np
import pytest
import torch

import workloads
from parity_util import codes
from test_gpu_ffn import MODES, _staged, compare_block_with_oracle

pytestmark = pytest.mark.gpu

SIZES = [200, 0, 57]   # a ragged group, an empty group, a sub-tile group
D, F = 128, 256


@pytest.fixture(scope="module")
def s3r():
    import stochastic_rounding_int8_gb300 as m
    m.lib()
    return m


def _offsets(sizes):
    return [0] + list(np.cumsum(sizes))


def _device_ops(s3r, inp, fmt):
    c = lambda t: t.cuda()
    return s3r.moe_forward_operands(c(inp.X), c(inp.W1), c(inp.W3), c(inp.W2), c(inp.a), c(inp.h1), c(inp.h3),
                                    code_format=fmt)


def _expert_ops(s3r, ops, e, r0, r1):
    return s3r.FFNOperands(ops.X8[r0:r1], ops.s_x[r0:r1], ops.A8[r0:r1], ops.s_a[r0:r1], ops.W1_8[e], ops.s_w1[e],
                           ops.W3_8[e], ops.s_w3[e], ops.W2_8[e], ops.s_w2[e], ops.h1[r0:r1], ops.h3[r0:r1])


@pytest.mark.parametrize("fmt", [0, 1], ids=["s8", "f16"])
@pytest.mark.parametrize("mode,ec", MODES)
def test_grouped_equals_staged_per_expert(s3r, fmt, mode, ec):
    inp = workloads.moe_inputs_sized(SIZES, D, F, seed=21)
    ops = _device_ops(s3r, inp, fmt)
    rm, ecm = getattr(s3r, "ROUND_" + mode), getattr(s3r, ec)
    dY = inp.dY.cuda()
    offs = _offsets(SIZES)
    st = s3r.new_status()
    g = s3r.ffn_backward(ops, dY, 0, rm, ecm, seed=9, status=st, group_offsets=offs)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for e in range(len(SIZES)):
        r0, r1 = offs[e], offs[e + 1]
        if r1 == r0:
            assert not g.dW1[e].any() and not g.dW3[e].any() and not g.dW2[e].any()
            continue
        ref = _staged(s3r, _expert_ops(s3r, ops, e, r0, r1), dY[r0:r1], r1 - r0, rm, ecm, 9,
                      tid_base=s3r.MOE_TID_STRIDE * e)
        torch.cuda.synchronize()
        assert torch.equal(g.dX[r0:r1], ref["dX"]), e
        assert torch.equal(g.dW1[e], ref["dW1"]) and torch.equal(g.dW3[e], ref["dW3"]), e
        assert torch.equal(g.dW2[e], ref["dW2"]), e


@pytest.mark.parametrize("fmt", [0, 1], ids=["s8", "f16"])
@pytest.mark.parametrize("mode,ec", [("S3R", "EC_TWO_WAY"), ("INDEP", "EC_NONE")])
def test_staged_experts_match_oracle(s3r, orc, fmt, mode, ec):
    inp = workloads.moe_inputs_sized(SIZES, D, F, seed=22)
    ops = _device_ops(s3r, inp, fmt)
    f = orc.from_torch_bf16
    ops_o = orc.moe_forward_operands(f(inp.X), f(inp.W1), f(inp.W3), f(inp.W2), f(inp.a))
    assert np.array_equal(codes(ops.W1_8), ops_o.W1_8) and np.array_equal(ops.s_w2.cpu().numpy(), ops_o.s_w2)
    rm, ecm = getattr(s3r, "ROUND_" + mode), getattr(s3r, ec)
    offs = _offsets(SIZES)
    h1, h3, dY = (f(t) for t in (inp.h1, inp.h3, inp.dY))
    for e in range(len(SIZES)):
        r0, r1 = offs[e], offs[e + 1]
        if r1 == r0:
            continue
        gpu = _staged(s3r, _expert_ops(s3r, ops, e, r0, r1), inp.dY.cuda()[r0:r1], r1 - r0, rm, ecm, 4,
                      tid_base=s3r.MOE_TID_STRIDE * e)
        torch.cuda.synchronize()
        compare_block_with_oracle(s3r, orc, gpu, ops_o.expert(e, r0, r1), h1[r0:r1], h3[r0:r1], dY[r0:r1],
                                  r1 - r0, mode, ec, 4, tid_base=orc.MOE_TID_STRIDE * e)
