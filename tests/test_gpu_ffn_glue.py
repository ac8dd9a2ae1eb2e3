"""GPU: the SwiGLU glue fused into the dA GEMM's epilogue (S3R_FFN_FUSE_GLUE).

ffn_backward with fuse_glue=True never stores dA: each 128 x 128 tile of it is
turned into dh1 and dh3, folded and quantized inside the GEMM that produced it
([S3R] §III-B, the threshold broadcast and the rounding inside the fusion that
makes the gradient; §IV-A, the SwiGLU block).  The dA values are the same fp32
bits either way, so the codes of dh1 and dh3 and their tile scales must equal
those of the separate SwiGLU quantizer bit for bit, and so must everything
that does not depend on the error partials; the partials are the same sums in
another order, so the corrected gradients agree to within fp32 rounding.
Element-by-element parity of the fused block with the oracle is in
test_gpu_ffn_oracle.py.
"""
import numpy as np
import pytest
import torch

import workloads
from parity_util import codes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def s3r():
    import stochastic_rounding_int8_gb300 as m
    m.lib()
    return m


def _run(s3r, ops, dY, S, rm, ec, seed, fuse):
    T, d = dY.shape
    F = ops.A8.shape[1]
    ws = torch.zeros(s3r.ffn_workspace_size(T, d, F, S, rm, ec), dtype=torch.uint8, device="cuda")
    st = s3r.new_status()
    g = s3r.ffn_backward(ops, dY, S, rm, ec, seed=seed, workspace=ws, status=st, fuse_glue=fuse)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return g, s3r.ffn_workspace_views(ws, T, d, F, S, round_mode=rm)


def _close(got, ref, what, rtol=1e-5):
    got = got.double().cpu()
    ref = ref.double().cpu()
    assert torch.isfinite(got).all(), what
    tol = rtol * ref.abs() + 1e-6 * float(ref.abs().max()) + 1e-30
    bad = (got - ref).abs() > tol
    assert not bool(bad.any()), f"{what}: {int(bad.sum())} of {bad.numel()} outside tolerance"


MODES = [("S3R", "EC_TWO_WAY"), ("S3R", "EC_DX_ONLY"), ("S3R", "EC_NONE"), ("S3R", "EC_DW_ONLY"),
         ("S3R_7BIT", "EC_TWO_WAY"), ("BCAST", "EC_TWO_WAY"), ("RTNE", "EC_NONE")]
SHAPES = [(1920, 520, 1416, 640), (2048, 256, 1288, 2048), (384, 128, 2048, 128)]


@pytest.mark.parametrize("T,d,F,S", SHAPES)
@pytest.mark.parametrize("rm,ec", MODES)
def test_fused_glue_equals_separate_quantizer(s3r, T, d, F, S, rm, ec):
    """Ragged shapes (F not a multiple of 128 or 256; a 256-wide tile whose
    second half lies past F; one row tile), every rounding mode the fusion
    takes and every correction mode."""
    rmode, emode = getattr(s3r, "ROUND_" + rm), getattr(s3r, ec)
    inp = workloads.ffn_inputs(T, d, F, S, seed=91 + T + F)
    c = lambda t: t.cuda()
    ops = s3r.ffn_forward_operands(c(inp.X), c(inp.W1), c(inp.W3), c(inp.W2), c(inp.a), c(inp.h1), c(inp.h3))
    dY = c(inp.dY)
    ref, rv = _run(s3r, ops, dY, S, rmode, emode, 5, False)
    got, gv = _run(s3r, ops, dY, S, rmode, emode, 5, True)
    for k in ("Q2", "Q1", "Q3"):
        assert np.array_equal(codes(gv[k]), codes(rv[k])), k
    for k in ("scale2", "scale1", "scale3"):
        assert torch.equal(gv[k], rv[k]), k
    assert torch.equal(got.dW2, ref.dW2), "dW2 (same launch, same tiles)"
    uses_partials = emode != s3r.EC_NONE and rmode != s3r.ROUND_RTNE
    for k in ("dX", "dW1", "dW3"):
        if uses_partials:
            _close(getattr(got, k), getattr(ref, k), k)
        else:
            assert torch.equal(getattr(got, k), getattr(ref, k)), k


def test_fused_glue_d2048_block_equals_separate(s3r):
    """The d=2048, F=5632, T=8192 block (S3R-EC two-way): every code and tile
    scale of Q1 and Q3 equal, the gradients within fp32 rounding; two calls
    in a row give the same result (no state left behind)."""
    T, d, F, S = 8192, 2048, 5632, 2048
    inp = workloads.ffn_inputs(T, d, F, S, seed=workloads.DATA_SEED + 1)
    c = lambda t: t.cuda()
    ops = s3r.ffn_forward_operands(c(inp.X), c(inp.W1), c(inp.W3), c(inp.W2), c(inp.a), c(inp.h1), c(inp.h3))
    dY = c(inp.dY)
    ref, rv = _run(s3r, ops, dY, S, s3r.ROUND_S3R, s3r.EC_TWO_WAY, 0, False)
    got, gv = _run(s3r, ops, dY, S, s3r.ROUND_S3R, s3r.EC_TWO_WAY, 0, True)
    again, av = _run(s3r, ops, dY, S, s3r.ROUND_S3R, s3r.EC_TWO_WAY, 0, True)
    for k in ("Q1", "Q3", "scale1", "scale3"):
        assert torch.equal(gv[k], rv[k]), k
        assert torch.equal(av[k], gv[k]), k
    for k in ("dX", "dW1", "dW3", "dW2"):
        _close(getattr(got, k), getattr(ref, k), k)
        assert torch.equal(getattr(again, k), getattr(got, k)), k


def test_fused_glue_nonfinite_gradient(s3r):
    """A NaN in dY makes its dA tiles non-finite: the fused glue reports
    S3R_ERR_NONFINITE, as the separate quantizer does."""
    T, d, F, S = 256, 128, 512, 256
    inp = workloads.ffn_inputs(T, d, F, S, seed=3)
    c = lambda t: t.cuda()
    ops = s3r.ffn_forward_operands(c(inp.X), c(inp.W1), c(inp.W3), c(inp.W2), c(inp.a), c(inp.h1), c(inp.h3))
    dY = c(inp.dY)
    dY[5, 7] = float("nan")
    ws = torch.zeros(s3r.ffn_workspace_size(T, d, F, S), dtype=torch.uint8, device="cuda")
    st = s3r.new_status()
    s3r.ffn_backward(ops, dY, S, workspace=ws, status=st, fuse_glue=True)
    torch.cuda.synchronize()
    assert int(st.item()) == -4   # S3R_ERR_NONFINITE
