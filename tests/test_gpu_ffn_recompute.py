"""GPU: ffn_backward forming the codes of a itself (S3R_FFN_RECOMPUTE_A).

With the flag the call makes A8 and s_a from h1 and h3 with the forward's
own kernel (swiglu_fwd_quantize) inside its workspace, so every gradient and
intermediate must equal a call given the A8 and s_a that swiglu_fwd_quantize
makes from the same h1 and h3, bit for bit: in every rounding mode, with int8
codes at rest widened inside the call, with the SwiGLU glue fused into the dA
GEMM, in grouped mode and with int8 codes on the mma.sync path.
Element-by-element parity of the block with the oracle is in
test_gpu_ffn_oracle.py.
"""
import dataclasses

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def s3r():
    import stochastic_rounding_int8_gb300 as m
    m.lib()
    return m


def _forward_a(s3r, ops, fmt):
    """ops with A8 and s_a from the forward's SwiGLU kernel (in `fmt`)."""
    _, A8, s_a = s3r.swiglu_fwd_quantize(ops.h1, ops.h3, keep_a=False, code_format=fmt)
    return dataclasses.replace(ops, A8=A8, s_a=s_a)


def _run(s3r, ops, dY, S, rm, ec, recompute, group_offsets=None, widen=False, fuse=False):
    T, d = dY.shape
    F = ops.h1.shape[1]
    fmt = s3r.CODES_S8_F16 if widen else s3r.code_format_of(ops.X8)
    flags = s3r.FFN_RECOMPUTE_A if recompute else 0
    if group_offsets is None:
        n = s3r.ffn_workspace_size(T, d, F, S, rm, ec, fmt, flags)
    else:
        n = s3r.grouped_workspace_size(group_offsets, d, F, rm, ec, fmt, flags)
    ws = torch.full((n,), 0x5A, dtype=torch.uint8, device="cuda")
    st = s3r.new_status()
    run_ops = dataclasses.replace(ops, A8=None, s_a=None) if recompute else ops
    g = s3r.ffn_backward(run_ops, dY, S, rm, ec, seed=7, workspace=ws, status=st, group_offsets=group_offsets,
                         widen_codes=widen, fuse_glue=fuse, recompute_a=recompute)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    if group_offsets is None:
        v = s3r.ffn_workspace_views(ws, T, d, F, S, round_mode=rm, code_format=fmt)
        views = {0: v}
    else:
        views = {e: s3r.ffn_workspace_views(ws, T, d, F, S, round_mode=rm, code_format=fmt,
                                            group_offsets=group_offsets, group=e)
                 for e in range(len(group_offsets) - 1) if group_offsets[e + 1] > group_offsets[e]}
    return g, views


def _same(got, ref, gv, rv, fuse=False):
    for k in ("dX", "dW1", "dW3", "dW2"):
        assert torch.equal(getattr(got, k), getattr(ref, k)), k
    keys = ("Q2", "scale2", "Q1", "scale1", "Q3", "scale3") + (() if fuse else ("dA",))
    assert set(gv) == set(rv)
    for e in gv:
        for k in keys:
            assert torch.equal(gv[e][k], rv[e][k]), (e, k)


def _dense(s3r, T, d, F, S, seed, fmt=None):
    inp = workloads.ffn_inputs(T, d, F, S, seed=seed)
    c = lambda t: t.cuda()
    kw = {} if fmt is None else {"code_format": fmt}
    ops = s3r.ffn_forward_operands(c(inp.X), c(inp.W1), c(inp.W3), c(inp.W2), c(inp.a), c(inp.h1), c(inp.h3), **kw)
    return ops, c(inp.dY)


MODES = [("S3R", "EC_TWO_WAY"), ("S3R", "EC_DX_ONLY"), ("S3R_7BIT", "EC_TWO_WAY"), ("INDEP", "EC_NONE"),
         ("RTNE", "EC_NONE")]


@pytest.mark.parametrize("rm,ec", MODES)
@pytest.mark.parametrize("T,d,F,S", [(2048, 512, 1536, 1024), (1920, 520, 1416, 640)])
def test_recomputed_a_equals_forward_a(s3r, rm, ec, T, d, F, S):
    rmode, emode = getattr(s3r, "ROUND_" + rm), getattr(s3r, ec)
    ops, dY = _dense(s3r, T, d, F, S, 23 + T + F)
    ops = _forward_a(s3r, ops, s3r.CODES_F16)
    ref, rv = _run(s3r, ops, dY, S, rmode, emode, False)
    got, gv = _run(s3r, ops, dY, S, rmode, emode, True)
    _same(got, ref, gv, rv)


def test_recomputed_a_with_widened_codes_and_fused_glue(s3r):
    """int8 codes at rest (the recomputed codes of a go straight into the fp16
    copies), and the SwiGLU glue fused into the dA GEMM."""
    T, d, F, S = 2048, 512, 1536, 1024
    ops, dY = _dense(s3r, T, d, F, S, 31)
    ops = _forward_a(s3r, ops, s3r.CODES_F16)
    ops8 = dataclasses.replace(ops, **{k: getattr(ops, k).to(torch.int8)
                                       for k in ("X8", "A8", "W1_8", "W3_8", "W2_8")})
    ref, rv = _run(s3r, ops, dY, S, s3r.ROUND_S3R, s3r.EC_TWO_WAY, False)
    got, gv = _run(s3r, ops8, dY, S, s3r.ROUND_S3R, s3r.EC_TWO_WAY, True, widen=True)
    _same(got, ref, gv, rv)
    ref, rv = _run(s3r, ops, dY, S, s3r.ROUND_S3R, s3r.EC_TWO_WAY, False, fuse=True)
    got, gv = _run(s3r, ops, dY, S, s3r.ROUND_S3R, s3r.EC_TWO_WAY, True, fuse=True)
    _same(got, ref, gv, rv, fuse=True)


def test_recomputed_a_grouped(s3r):
    d, F = 256, 384
    mi = workloads.moe_inputs_sized([700, 0, 129, 1024, 64], d, F, seed=37)
    c = lambda t: t.cuda()
    ops = s3r.moe_forward_operands(c(mi.X), c(mi.W1), c(mi.W3), c(mi.W2), c(mi.a), c(mi.h1), c(mi.h3))
    ops = _forward_a(s3r, ops, s3r.CODES_F16)
    offs = list(mi.offsets)
    dY = c(mi.dY)
    ref, rv = _run(s3r, ops, dY, 0, s3r.ROUND_S3R, s3r.EC_TWO_WAY, False, group_offsets=offs)
    got, gv = _run(s3r, ops, dY, 0, s3r.ROUND_S3R, s3r.EC_TWO_WAY, True, group_offsets=offs)
    _same(got, ref, gv, rv)


def test_recomputed_a_int8_codes(s3r):
    """int8 codes on the mma.sync path: the recomputed codes of a are int8 too."""
    T, d, F, S = 256, 128, 384, 256
    ops, dY = _dense(s3r, T, d, F, S, 3, fmt=s3r.CODES_S8)
    ops = _forward_a(s3r, ops, s3r.CODES_S8)
    ref, rv = _run(s3r, ops, dY, S, s3r.ROUND_S3R, s3r.EC_TWO_WAY, False)
    got, gv = _run(s3r, ops, dY, S, s3r.ROUND_S3R, s3r.EC_TWO_WAY, True)
    _same(got, ref, gv, rv)
