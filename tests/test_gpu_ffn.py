"""GPU parity: the SwiGLU FFN block backward.

1. ffn_backward equals the same steps called one by one (bit for bit).
2. The steps match the oracle's chain.  The first stage (W2) is compared
   directly.  In the second stage the gate/up gradients come from the fp32
   dA, whose last bits depend on the summation order, so a code may differ by
   one step where the oracle's decision was a near tie; the test checks that
   every such difference is a near tie and adds its exact linear effect
   (through the correction and both products) before comparing dX, dW1, dW3.
ffn_backward itself at full size, element by element against the oracle, is
in test_gpu_ffn_oracle.py.
"""
import numpy as np
import pytest
import torch

import workloads
from parity_util import assert_close_mag, codes, dw_magnitude, dx_magnitude, expand_tiles, near_tie_flips, projection

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def s3r():
    import stochastic_rounding_int8_gb300 as m
    m.lib()
    return m


def _staged(s3r, ops, dY, S, rm, ec, seed, tid_base=0):
    """The block backward as separate library calls (same order as ffn_backward);
    the three linears use tensor ids tid_base + (0, 1, 2)."""
    T, d = dY.shape
    F = ops.A8.shape[1]
    out = {}
    indep = rm == s3r.ROUND_INDEP
    shared = rm in (s3r.ROUND_S3R, s3r.ROUND_S3R_7BIT, s3r.ROUND_BCAST)
    ecm = ec if shared else s3r.EC_NONE
    cf = s3r.code_format_of(ops.X8)
    if shared:
        q2, _ = s3r.s3r_quantize_ex(dY, ops.s_a, ops.s_w2, rm, S, seed=seed, tensor_id=tid_base + s3r.TID_W2,
                                    code_format=cf)
    elif indep:
        q2 = s3r.indep_sr_quantize(dY, ops.s_a, ops.s_w2, seed, tid_base + s3r.TID_W2, code_format=cf)
        out["q2r"] = s3r.indep_sr_quantize(dY, ops.s_a, ops.s_w2, seed, tid_base + s3r.TID_W2 + s3r.RHS_ID_OFFSET,
                                           code_format=cf)
    else:
        Q, sc = s3r.rtne_quantize(dY, s3r.AXIS_TILE, s_x=ops.s_a, s_w=ops.s_w2, code_format=cf)
        q2 = s3r.Quantized(Q, sc)
    ec2 = s3r.s3r_ec_correct(q2, T, d, S, ops.W2_8, ops.A8, ecm) if ecm else None
    dA = s3r.int8_gemm_dx(q2.Q, q2.tile_scale, ops.W2_8, ops.s_a, ecm, ec2, S)
    q2w = out.get("q2r", q2)
    dW2 = s3r.int8_gemm_dw(ops.A8, q2w.Q, q2w.tile_scale, ops.s_w2, ecm, ec2, S)
    q1, q3 = s3r.swiglu_quantize(dA, ops.h1, ops.h3, ops.s_x, ops.s_w1, ops.s_w3, rm, seed, tid_base + s3r.TID_W1,
                                 tid_base + s3r.TID_W3, code_format=cf, S=S)
    if indep:
        out["q1r"], out["q3r"] = s3r.swiglu_quantize(dA, ops.h1, ops.h3, ops.s_x, ops.s_w1, ops.s_w3, rm, seed,
                                                     tid_base + s3r.TID_W1 + s3r.RHS_ID_OFFSET,
                                                     tid_base + s3r.TID_W3 + s3r.RHS_ID_OFFSET, code_format=cf)
    ec1 = s3r.s3r_ec_correct(q1, T, F, S, ops.W1_8, ops.X8, ecm) if ecm else None
    ec3 = s3r.s3r_ec_correct(q3, T, F, S, ops.W3_8, ops.X8, ecm) if ecm else None
    dX = s3r.int8_gemm_dx_sum([(q1.Q, q1.tile_scale, ops.W1_8, ec1), (q3.Q, q3.tile_scale, ops.W3_8, ec3)],
                              ops.s_x, ecm, S)
    q1w, q3w = out.get("q1r", q1), out.get("q3r", q3)
    dW1 = s3r.int8_gemm_dw(ops.X8, q1w.Q, q1w.tile_scale, ops.s_w1, ecm, ec1, S)
    dW3 = s3r.int8_gemm_dw(ops.X8, q3w.Q, q3w.tile_scale, ops.s_w3, ecm, ec3, S)
    out.update(q2=q2, dA=dA, dW2=dW2, q1=q1, q3=q3, dX=dX, dW1=dW1, dW3=dW3)
    return out


def _device_ops(s3r, inp, fmt=1):
    c = lambda t: t.cuda()
    return s3r.ffn_forward_operands(c(inp.X), c(inp.W1), c(inp.W3), c(inp.W2), c(inp.a), c(inp.h1), c(inp.h3),
                                    code_format=fmt)


def _oracle_ops(orc, inp):
    f = orc.from_torch_bf16
    return orc.ffn_forward_operands(f(inp.X), f(inp.W1), f(inp.W3), f(inp.W2), f(inp.a))


MODES = [("S3R", "EC_TWO_WAY"), ("S3R", "EC_DX_ONLY"), ("S3R", "EC_NONE"), ("INDEP", "EC_NONE"), ("RTNE", "EC_NONE"),
         ("S3R_7BIT", "EC_TWO_WAY"), ("BCAST", "EC_TWO_WAY"), ("S3R", "EC_DW_ONLY")]
ORACLE_MODE = {"S3R_7BIT": "S3R7"}   # oracle constant names that differ from the library's


def _omode(orc, mode):
    return getattr(orc, ORACLE_MODE.get(mode, mode))


@pytest.mark.parametrize("fmt", [0, 1], ids=["s8", "f16"])
@pytest.mark.parametrize("mode,ec", MODES)
def test_ffn_backward_equals_staged_calls(s3r, fmt, mode, ec):
    inp = workloads.ffn_inputs(512, 256, 384, 256, seed=7)
    ops = _device_ops(s3r, inp, fmt)
    rm, ecm = getattr(s3r, "ROUND_" + mode), getattr(s3r, ec)
    st = s3r.new_status()
    g = s3r.ffn_backward(ops, inp.dY.cuda(), 256, rm, ecm, seed=9, status=st)
    ref = _staged(s3r, ops, inp.dY.cuda(), 256, rm, ecm, seed=9)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for k in ("dX", "dW1", "dW3", "dW2"):
        assert torch.equal(getattr(g, k), ref[k]), k


def _forward_ops_bit_exact(ops_g, ops_o):
    for name in ("X8", "A8", "W1_8", "W3_8", "W2_8"):
        assert np.array_equal(codes(getattr(ops_g, name)), getattr(ops_o, name)), name
    for name in ("s_x", "s_a", "s_w1", "s_w3", "s_w2"):
        assert np.array_equal(getattr(ops_g, name).cpu().numpy(), getattr(ops_o, name)), name


def _flip_effect(D, W8, X8, s_x, s_w, S, ecm, orc):
    """Exact change of (dX, dW) when the dequantized operand changes by D."""
    Dx = D - projection(D, S) if ecm in (orc.EC_DX_ONLY, orc.EC_TWO_WAY) else D
    Dw = D - projection(D, S) if ecm in (orc.EC_TWO_WAY, orc.EC_DW_ONLY) else D
    ddx = (Dx @ W8.astype(np.float64).T) / s_x[:, None].astype(np.float64)
    ddw = (X8.astype(np.float64).T @ Dw) / s_w[None, :].astype(np.float64)
    return ddx, ddw


def _thresholds(orc, mode, T, N, seed, tid, S=0):
    if mode == "S3R":
        return np.array([orc.token_threshold(t, seed, tid) for t in range(T)])[:, None]
    if mode == "S3R_7BIT":
        return np.array([orc.token_threshold7(t, seed, tid) for t in range(T)])[:, None]
    if mode == "BCAST":
        return np.array([orc.example_threshold(t // S if S else 0, seed, tid) for t in range(T)])[:, None]
    if mode == "INDEP":
        return np.array([[orc.element_threshold(t * N + n, seed, tid) for n in range(N)] for t in range(T)])
    return 0.5


def _tile_amax(g):
    """Per-128x128-tile absmax of g [T, F] (ragged edges included)."""
    T, F = g.shape
    nt, nf = -(-T // 128), -(-F // 128)
    out = np.zeros((nt, nf), dtype=np.float32)
    for i in range(nt):
        for j in range(nf):
            out[i, j] = np.abs(g[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]).max()
    return out


def compare_block_with_oracle(s3r, orc, gpu, ops_o, h1, h3, dY, S, mode, ec, seed, tid_base=0):
    """Checks the staged GPU outputs `gpu` of one block (or one expert's
    group) against the oracle: stage 1 (W2) directly; stage 2 allowing only
    near-tie code flips, whose exact linear effect is added to the oracle."""
    T = dY.shape[0]
    F = ops_o.A8.shape[1]
    omode, oec = _omode(orc, mode), getattr(orc, ec)
    ref = orc.ffn_backward(ops_o, h1, h3, dY, S, mode=omode, ec_mode=oec, seed=seed, tid_base=tid_base)
    ecx = oec if omode in orc.SHARED else orc.EC_NONE
    dx_ec = ecx in (orc.EC_DX_ONLY, orc.EC_TWO_WAY)
    dw_ec = ecx in (orc.EC_TWO_WAY, orc.EC_DW_ONLY)
    # stage 1: codes exact, dA and dW2 within the fp32 bound
    assert np.array_equal(codes(gpu["q2"].Q), ref.w2.Q)
    w2 = ref.w2
    mdx = dx_magnitude(w2.Q, w2.delta, ops_o.W2_8, ops_o.s_a,
                       *( (w2.eps, w2.rowsum, w2.v, S) if dx_ec else (None, None, None, None)))
    assert_close_mag(gpu["dA"].cpu().numpy(), w2.dX, mdx, "dA")
    Qw2 = w2.Q_rhs if omode == orc.INDEP else w2.Q
    dw2 = w2.delta_rhs if omode == orc.INDEP else w2.delta
    mdw = dw_magnitude(ops_o.A8, Qw2, dw2, ops_o.s_w2,
                       *((w2.colmean, w2.mu, w2.xsum, w2.p) if dw_ec else (None,) * 4))
    assert_close_mag(gpu["dW2"].cpu().numpy(), w2.dW, mdw, "dW2")
    # stage 2: near-tie flips only; their exact effect added to the oracle
    exp_dX = ref.dX.copy()
    exp = {"dW1": ref.dW1.copy(), "dW3": ref.dW3.copy()}
    mags_dx = np.zeros_like(ref.dX)
    mags = {}
    for name, lb, dh, W8, s_w, tid in (("dW1", ref.w1, ref.dh1, ops_o.W1_8, ops_o.s_w1, tid_base + orc.TID_W1),
                                       ("dW3", ref.w3, ref.dh3, ops_o.W3_8, ops_o.s_w3, tid_base + orc.TID_W3)):
        q = gpu["q1" if name == "dW1" else "q3"]
        Qg, dg = codes(q.Q), q.tile_scale.cpu().numpy()
        g = ((ops_o.s_x[:, None] * dh).astype(np.float32) * s_w[None, :]).astype(np.float32)
        inv = np.vectorize(lambda a: np.float32(orc.inv127_rz(float(a))))(_tile_amax(g)).astype(np.float32)
        y = (g * expand_tiles(inv, T, F).astype(np.float32)).astype(np.float32)
        near_tie_flips(Qg, lb.Q, y, _thresholds(orc, mode, T, F, seed, tid, S))
        D = expand_tiles(dg, T, F) * Qg - expand_tiles(lb.delta, T, F) * lb.Q
        ddx, ddw = _flip_effect(D, W8, ops_o.X8, ops_o.s_x, s_w, S, ecx, orc)
        exp_dX += ddx
        if omode == orc.INDEP:
            qr = gpu["q1r" if name == "dW1" else "q3r"]
            Qr, dr = codes(qr.Q), qr.tile_scale.cpu().numpy()
            near_tie_flips(Qr, lb.Q_rhs, y, _thresholds(orc, mode, T, F, seed, tid + orc.RHS_ID_OFFSET))
            Dr = expand_tiles(dr, T, F) * Qr - expand_tiles(lb.delta_rhs, T, F) * lb.Q_rhs
            _, ddw = _flip_effect(Dr, W8, ops_o.X8, ops_o.s_x, s_w, S, ecx, orc)
        exp[name] += ddw
        if dx_ec:
            mags_dx += dx_magnitude(lb.Q, lb.delta, W8, ops_o.s_x, lb.eps, lb.rowsum, lb.v, S)
        else:
            mags_dx += dx_magnitude(lb.Q, lb.delta, W8, ops_o.s_x)
        Qw = lb.Q_rhs if omode == orc.INDEP else lb.Q
        dw_ = lb.delta_rhs if omode == orc.INDEP else lb.delta
        mags[name] = dw_magnitude(ops_o.X8, Qw, dw_, s_w,
                                  *((lb.colmean, lb.mu, lb.xsum, lb.p) if dw_ec else (None,) * 4))
    assert_close_mag(gpu["dX"].cpu().numpy(), exp_dX, mags_dx, "dX")
    assert_close_mag(gpu["dW1"].cpu().numpy(), exp["dW1"], mags["dW1"], "dW1")
    assert_close_mag(gpu["dW3"].cpu().numpy(), exp["dW3"], mags["dW3"], "dW3")


@pytest.mark.parametrize("fmt", [0, 1], ids=["s8", "f16"])
@pytest.mark.parametrize("mode,ec", MODES)
def test_ffn_staged_matches_oracle(s3r, orc, fmt, mode, ec):
    T, d, F, S = 256, 128, 384, 128
    inp = workloads.ffn_inputs(T, d, F, S, seed=11)
    ops_g = _device_ops(s3r, inp, fmt)
    ops_o = _oracle_ops(orc, inp)
    _forward_ops_bit_exact(ops_g, ops_o)
    rm, ecm = getattr(s3r, "ROUND_" + mode), getattr(s3r, ec)
    seed = 5
    gpu = _staged(s3r, ops_g, inp.dY.cuda(), S, rm, ecm, seed)
    torch.cuda.synchronize()
    h1, h3, dY = (orc.from_torch_bf16(t) for t in (inp.h1, inp.h3, inp.dY))
    compare_block_with_oracle(s3r, orc, gpu, ops_o, h1, h3, dY, S, mode, ec, seed)
