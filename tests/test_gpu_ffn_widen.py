"""GPU: ffn_backward on int8 operand codes widened inside the call (S3R_CODES_S8_F16).

The five operand code tensors (X8, A8, W1_8, W3_8, W2_8) are the same
integers whether they are held as int8 or as fp16, and the widened call runs
the fp16-code block on fp16 copies of them, so every gradient and every
intermediate must equal the fp16-code call's bit for bit: the codes, tile
scales and dA in the workspace, dX, dW1, dW3 and dW2.  Element-by-element
parity of the fp16-code block with the oracle is in test_gpu_ffn_oracle.py.
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

CODE_FIELDS = ("X8", "A8", "W1_8", "W3_8", "W2_8")


@pytest.fixture(scope="module")
def s3r():
    import stochastic_rounding_int8_gb300 as m
    m.lib()
    return m


def _as_int8(s3r, ops, misalign=False):
    """The same operands with int8 codes; misalign: each code tensor starts one
    byte into its buffer (the widening then takes its element path)."""
    def conv(t):
        q = t.to(torch.int8)
        if not misalign:
            return q
        buf = torch.empty(q.numel() + 1, dtype=torch.int8, device=q.device)
        view = buf[1:].view(q.shape)
        view.copy_(q)
        return view
    return s3r.FFNOperands(**{k: (conv(getattr(ops, k)) if k in CODE_FIELDS else getattr(ops, k))
                              for k in s3r.FFNOperands.__dataclass_fields__})


def _run(s3r, ops, dY, S, rm, ec, seed, widen, group_offsets=None, fuse=False):
    T, d = dY.shape
    F = ops.A8.shape[1]
    fmt = s3r.CODES_S8_F16 if widen else s3r.CODES_F16
    if group_offsets is None:
        n = s3r.ffn_workspace_size(T, d, F, S, rm, ec, fmt)
    else:
        n = s3r.grouped_workspace_size(group_offsets, d, F, rm, ec, fmt)
    ws = torch.full((n,), 0xA5, dtype=torch.uint8, device="cuda")
    st = s3r.new_status()
    g = s3r.ffn_backward(ops, dY, S, rm, ec, seed=seed, workspace=ws, status=st, widen_codes=widen,
                         group_offsets=group_offsets, fuse_glue=fuse)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    if group_offsets is None:
        views = s3r.ffn_workspace_views(ws, T, d, F, S, round_mode=rm, code_format=fmt)
    else:
        views = {e: s3r.ffn_workspace_views(ws, T, d, F, S, round_mode=rm, code_format=fmt,
                                            group_offsets=group_offsets, group=e)
                 for e in range(len(group_offsets) - 1) if group_offsets[e + 1] > group_offsets[e]}
    return g, views


def _same(got, ref, gv, rv, fuse=False):
    for k in ("dX", "dW1", "dW3", "dW2"):
        assert torch.equal(getattr(got, k), getattr(ref, k)), k
    keys = ("Q2", "scale2", "Q1", "scale1", "Q3", "scale3") + (() if fuse else ("dA",))
    for k in keys:
        assert torch.equal(gv[k], rv[k]), k


MODES = [("S3R", "EC_TWO_WAY"), ("S3R", "EC_DX_ONLY"), ("S3R", "EC_DW_ONLY"), ("S3R_7BIT", "EC_TWO_WAY"),
         ("INDEP", "EC_NONE"), ("RTNE", "EC_NONE")]


@pytest.mark.parametrize("rm,ec", MODES)
@pytest.mark.parametrize("T,d,F,S,misalign", [(2048, 512, 1536, 1024, False), (1920, 520, 1416, 640, True)])
def test_widened_equals_fp16_codes(s3r, rm, ec, T, d, F, S, misalign):
    """Several tiles per CTA in both mixed GEMM launches; a ragged block whose
    int8 codes start one byte into their buffers."""
    rmode, emode = getattr(s3r, "ROUND_" + rm), getattr(s3r, ec)
    inp = workloads.ffn_inputs(T, d, F, S, seed=17 + T + F)
    c = lambda t: t.cuda()
    ops = s3r.ffn_forward_operands(c(inp.X), c(inp.W1), c(inp.W3), c(inp.W2), c(inp.a), c(inp.h1), c(inp.h3))
    dY = c(inp.dY)
    ops8 = _as_int8(s3r, ops, misalign)
    assert all(getattr(ops8, k).dtype == torch.int8 for k in CODE_FIELDS)
    ref, rv = _run(s3r, ops, dY, S, rmode, emode, 3, False)
    got, gv = _run(s3r, ops8, dY, S, rmode, emode, 3, True)
    _same(got, ref, gv, rv)


def test_widened_d2048_block_and_fused_glue(s3r):
    """The d=2048, F=5632, T=8192 block, S3R-EC two-way: equal to the fp16-code
    call, also with the SwiGLU glue fused into the dA GEMM."""
    T, d, F, S = 8192, 2048, 5632, 2048
    inp = workloads.ffn_inputs(T, d, F, S, seed=workloads.DATA_SEED + 1)
    c = lambda t: t.cuda()
    ops = s3r.ffn_forward_operands(c(inp.X), c(inp.W1), c(inp.W3), c(inp.W2), c(inp.a), c(inp.h1), c(inp.h3))
    dY = c(inp.dY)
    ops8 = _as_int8(s3r, ops)
    for fuse in (False, True):
        ref, rv = _run(s3r, ops, dY, S, s3r.ROUND_S3R, s3r.EC_TWO_WAY, 0, False, fuse=fuse)
        got, gv = _run(s3r, ops8, dY, S, s3r.ROUND_S3R, s3r.EC_TWO_WAY, 0, True, fuse=fuse)
        _same(got, ref, gv, rv, fuse)


def test_widened_grouped_equals_fp16_codes(s3r):
    """Grouped mode on ragged experts (one of them empty): stacked int8 weight
    codes widened once for all experts."""
    d, F = 256, 384
    sizes = [700, 0, 129, 1024, 64]
    mi = workloads.moe_inputs_sized(sizes, d, F, seed=29)
    c = lambda t: t.cuda()
    ops = s3r.moe_forward_operands(c(mi.X), c(mi.W1), c(mi.W3), c(mi.W2), c(mi.a), c(mi.h1), c(mi.h3))
    dY = c(mi.dY)
    offs = list(mi.offsets)
    ops8 = _as_int8(s3r, ops)
    ref, rv = _run(s3r, ops, dY, 0, s3r.ROUND_S3R, s3r.EC_TWO_WAY, 4, False, group_offsets=offs)
    got, gv = _run(s3r, ops8, dY, 0, s3r.ROUND_S3R, s3r.EC_TWO_WAY, 4, True, group_offsets=offs)
    for k in ("dX", "dW1", "dW3", "dW2"):
        assert torch.equal(getattr(got, k), getattr(ref, k)), k
    assert set(gv) == set(rv)
    for e in gv:
        for k in ("Q2", "scale2", "Q1", "scale1", "Q3", "scale3", "dA"):
            assert torch.equal(gv[e][k], rv[e][k]), (e, k)


def test_widening_is_exact(s3r):
    """Every int8 value, at every position of a 16-byte group and in the
    element tail: a block whose operands hold all 256 codes gives the same
    result as the fp16-code call (the widening itself is not exported)."""
    T, d, F, S = 256, 128, 256, 256
    inp = workloads.ffn_inputs(T, d, F, S, seed=5)
    c = lambda t: t.cuda()
    ops = s3r.ffn_forward_operands(c(inp.X), c(inp.W1), c(inp.W3), c(inp.W2), c(inp.a), c(inp.h1), c(inp.h3))
    full = torch.arange(-128, 128, dtype=torch.float16, device="cuda")
    for k in CODE_FIELDS:
        t = getattr(ops, k)
        flat = t.view(-1)
        flat[:256] = full
        flat[-256:] = full.flip(0)
    dY = c(inp.dY)
    ref, rv = _run(s3r, ops, dY, S, s3r.ROUND_S3R, s3r.EC_TWO_WAY, 1, False)
    for misalign in (False, True):
        got, gv = _run(s3r, _as_int8(s3r, ops, misalign), dY, S, s3r.ROUND_S3R, s3r.EC_TWO_WAY, 1, True)
        _same(got, ref, gv, rv)
