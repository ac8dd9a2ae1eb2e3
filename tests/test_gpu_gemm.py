"""GPU parity: the INT8 backward GEMMs.

The int32 partial of every 128-wide contraction block is bit-exact against
brute force; the rescaled and corrected fp32 outputs match the fp64 oracle
within the fp32 bound.  Includes the full-size activation- and weight-gradient
GEMMs of the d=2048 / F=5632 / T=8192 FFN block on sampled rows.
"""
import numpy as np
import pytest
import torch

import workloads
from parity_util import assert_close_mag, codes, dw_magnitude, dx_magnitude

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def s3r():
    import stochastic_rounding_int8_gb300 as m
    m.lib()
    return m


FMTS = pytest.mark.parametrize("fmt", [0, 1], ids=["s8", "f16"])


def _i8(rng, *shape):
    return rng.integers(-127, 128, size=shape).astype(np.int8)


def _dev(a, fmt):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return (t.to(torch.float16) if fmt else t).cuda()


@FMTS
@pytest.mark.parametrize("T,N,K", [(256, 1024, 512), (130, 136, 70), (1, 16, 1), (300, 384, 257), (64, 1000, 33),
                                   (129, 4096, 300)])
def test_dx_blocks_bit_exact(s3r, orc, fmt, T, N, K):
    rng = np.random.default_rng(T * N + K)
    Q, W8 = _i8(rng, T, N), _i8(rng, K, N)
    Q[0, :] = 127
    W8[0, :] = 127          # the largest block sum, 128 * 127^2
    W8[-1, :] = -127
    got = s3r.debug_dx_blocks(_dev(Q, fmt), _dev(W8, fmt)).cpu().numpy()
    ref = orc.dx_blocks(Q, W8, np.arange(T))
    assert np.array_equal(got, ref)


@FMTS
@pytest.mark.parametrize("T,K,N", [(256, 512, 1024), (130, 72, 136), (1, 8, 16), (300, 256, 384), (1000, 40, 64),
                                   (4096, 136, 200)])
def test_dw_blocks_bit_exact(s3r, orc, fmt, T, K, N):
    rng = np.random.default_rng(T + 3 * N + K)
    X8, Q = _i8(rng, T, K), _i8(rng, T, N)
    X8[:, 0] = -127
    Q[:, 0] = 127
    got = s3r.debug_dw_blocks(_dev(X8, fmt), _dev(Q, fmt)).cpu().numpy()
    ref = orc.dw_blocks(X8, Q, np.arange(K))
    assert np.array_equal(got, ref)


def _linear(orc, T, K, N, S, seed):
    inp = workloads.linear_inputs(T, K, N, S, seed=seed)
    X, W, G = (orc.from_torch_bf16(t) for t in (inp.X, inp.W, inp.dY))
    X8, s_x = orc.rtne_operand(X, 0)
    W8, s_w = orc.rtne_operand(W, 1)
    return inp, G, X8, s_x, W8, s_w


@FMTS
@pytest.mark.parametrize("ec_name", ["EC_NONE", "EC_DX_ONLY", "EC_TWO_WAY", "EC_DW_ONLY"])
@pytest.mark.parametrize("T,K,N,S", [(256, 512, 1024, 256), (512, 200, 384, 128), (300, 136, 264, 300)])
def test_linear_backward_parity(s3r, orc, fmt, ec_name, T, K, N, S):
    """dX and dW of one linear layer (the tiny-linear workload and ragged
    variants) through quantize -> correction -> both GEMMs."""
    inp, G, X8, s_x, W8, s_w = _linear(orc, T, K, N, S, seed=T + K + N)
    ec_mode = getattr(orc, ec_name)      # the oracle's constant
    ec_lib = getattr(s3r, ec_name)       # the library's
    ref = orc.linear_backward(G, X8, s_x, W8, s_w, S, mode=orc.S3R, ec_mode=ec_mode, seed=11, tensor_id=0)
    c = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    q = s3r.s3r_quantize(inp.dY.cuda(), c(s_x), c(s_w), seed=11, tensor_id=0, code_format=fmt)
    ec = s3r.s3r_ec_correct(q, T, N, S, _dev(W8, fmt), _dev(X8, fmt), ec_mode=ec_lib) if ec_lib else None
    dX = s3r.int8_gemm_dx(q.Q, q.tile_scale, _dev(W8, fmt), c(s_x), ec_lib, ec, S)
    dW = s3r.int8_gemm_dw(_dev(X8, fmt), q.Q, q.tile_scale, c(s_w), ec_lib, ec, S)
    torch.cuda.synchronize()
    assert np.array_equal(codes(q.Q), ref.Q)
    if ec_mode in (orc.EC_DX_ONLY, orc.EC_TWO_WAY):
        mdx = dx_magnitude(ref.Q, ref.delta, W8, s_x, ref.eps, ref.rowsum, ref.v, S)
    else:
        mdx = dx_magnitude(ref.Q, ref.delta, W8, s_x)
    assert_close_mag(dX.cpu().numpy(), ref.dX, mdx, "dX")
    if ec_mode in (orc.EC_TWO_WAY, orc.EC_DW_ONLY):
        mdw = dw_magnitude(X8, ref.Q, ref.delta, s_w, ref.colmean, ref.mu, ref.xsum, ref.p)
    else:
        mdw = dw_magnitude(X8, ref.Q, ref.delta, s_w)
    assert_close_mag(dW.cpu().numpy(), ref.dW, mdw, "dW")


@FMTS
def test_dx_accumulate(s3r, orc, fmt):
    rng = np.random.default_rng(1)
    T, N, K = 256, 256, 128
    Q, W8 = _i8(rng, T, N), _i8(rng, K, N)
    sc = (rng.random((2, 2)) + 0.5).astype(np.float32)
    c = lambda a: torch.from_numpy(a).cuda()
    base = torch.randn(T, K, device="cuda")
    out = base.clone()
    s3r.int8_gemm_dx(_dev(Q, fmt), c(sc), _dev(W8, fmt), dX=out, accumulate=True)
    fresh = s3r.int8_gemm_dx(_dev(Q, fmt), c(sc), _dev(W8, fmt))
    torch.cuda.synchronize()
    assert torch.allclose(out, base + fresh, rtol=1e-6, atol=1e-6)


@FMTS
@pytest.mark.parametrize("ec_name", ["EC_NONE", "EC_DX_ONLY"])
@pytest.mark.parametrize("T,K,N,S", [(256, 512, 1024, 256), (384, 200, 264, 128), (300, 136, 384, 300)])
def test_dx_sum_parity(s3r, orc, fmt, ec_name, T, K, N, S):
    """Input gradient of a layer that feeds two linears (X -> W1 and X -> W3 of
    the SwiGLU block): dX = dX1 + dX3, against the sum of the oracle's terms,
    and against two accumulating int8_gemm_dx calls."""
    inp1, G1, X8, s_x, W1_8, s_w1 = _linear(orc, T, K, N, S, seed=T + 1)
    inp3, G3, _, _, W3_8, s_w3 = _linear(orc, T, K, N, S, seed=T + 3)
    ec_mode = getattr(orc, ec_name)
    r1 = orc.linear_backward(G1, X8, s_x, W1_8, s_w1, S, mode=orc.S3R, ec_mode=ec_mode, seed=4, tensor_id=1)
    r3 = orc.linear_backward(G3, X8, s_x, W3_8, s_w3, S, mode=orc.S3R, ec_mode=ec_mode, seed=4, tensor_id=2)
    c = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    terms, qs = [], []
    for inp, W8, s_w, tid in ((inp1, W1_8, s_w1, 1), (inp3, W3_8, s_w3, 2)):
        q = s3r.s3r_quantize(inp.dY.cuda(), c(s_x), c(s_w), seed=4, tensor_id=tid, code_format=fmt)
        ec = s3r.s3r_ec_correct(q, T, N, S, _dev(W8, fmt), _dev(X8, fmt), ec_mode=ec_mode) if ec_mode else None
        terms.append((q.Q, q.tile_scale, _dev(W8, fmt), ec))
        qs.append(q)
    dX = s3r.int8_gemm_dx_sum(terms, c(s_x), ec_mode, S)
    two = s3r.int8_gemm_dx(*terms[0][:3], c(s_x), ec_mode, terms[0][3], S)
    s3r.int8_gemm_dx(*terms[1][:3], c(s_x), ec_mode, terms[1][3], S, dX=two, accumulate=True)
    torch.cuda.synchronize()
    assert np.array_equal(codes(qs[0].Q), r1.Q) and np.array_equal(codes(qs[1].Q), r3.Q)
    args = lambda r, W8: (r.Q, r.delta, W8, s_x) + ((r.eps, r.rowsum, r.v, S) if ec_mode else ())
    mag = dx_magnitude(*args(r1, W1_8)) + dx_magnitude(*args(r3, W3_8))
    assert_close_mag(dX.cpu().numpy(), r1.dX + r3.dX, mag, "dX1 + dX3")
    assert_close_mag(dX.cpu().numpy(), two.cpu().numpy().astype(np.float64), mag, "fused vs two calls")


def test_dx_sum_accumulate_and_single_term(s3r):
    rng = np.random.default_rng(2)
    T, N, K = 256, 256, 384
    Q, W8 = _i8(rng, T, N), _i8(rng, K, N)
    sc = (rng.random((2, 2)) + 0.5).astype(np.float32)
    c = lambda a: torch.from_numpy(a).cuda()
    one = s3r.int8_gemm_dx_sum([(_dev(Q, 1), c(sc), _dev(W8, 1), None)])
    ref = s3r.int8_gemm_dx(_dev(Q, 1), c(sc), _dev(W8, 1))
    base = torch.randn(T, K, device="cuda")
    out = base.clone()
    s3r.int8_gemm_dx_sum([(_dev(Q, 1), c(sc), _dev(W8, 1), None)], dX=out, accumulate=True)
    torch.cuda.synchronize()
    assert torch.equal(one, ref)
    assert torch.allclose(out, base + ref, rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("fmt,ec_name", [(1, "EC_DX_ONLY"), (1, "EC_TWO_WAY"), (0, "EC_TWO_WAY")])
def test_ffn_w2_gemms_full_size_sampled(s3r, orc, fmt, ec_name):
    """The W2 linear of the d=2048, F=5632, T=8192 (4 x 2048) SwiGLU block at
    full size through the standalone int8_gemm_dx / int8_gemm_dw launches
    (ffn_backward's own mixed launches are compared in
    test_gpu_ffn_oracle.py): dA = dX of W2 [8192, 5632] and dW2 [5632, 2048],
    checked on 48 sampled rows each."""
    T, d, F, S = 8192, 2048, 5632, 2048
    inp = workloads.ffn_inputs(T, d, F, S, seed=workloads.DATA_SEED + 1)
    A = orc.from_torch_bf16(inp.a)
    W2 = orc.from_torch_bf16(inp.W2)
    G = orc.from_torch_bf16(inp.dY)
    A8, s_a = orc.rtne_operand(A, 0)
    W8, s_w = orc.rtne_operand(W2, 1)
    ec_mode = getattr(orc, ec_name)
    rng = np.random.default_rng(0)
    rows = np.sort(np.concatenate([[0, T - 1], rng.choice(T, 46, replace=False)]))
    krows = np.sort(np.concatenate([[0, F - 1], rng.choice(F, 46, replace=False)]))
    ref = orc.linear_backward(G, A8, s_a, W8, s_w, S, mode=orc.S3R, ec_mode=ec_mode, seed=0, tensor_id=0,
                              rows=rows, krows=krows)
    c = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    q = s3r.s3r_quantize(inp.dY.cuda(), c(s_a), c(s_w), seed=0, tensor_id=0, code_format=fmt)
    ec = s3r.s3r_ec_correct(q, T, d, S, _dev(W8, fmt), _dev(A8, fmt), ec_mode=ec_mode)
    dA = s3r.int8_gemm_dx(q.Q, q.tile_scale, _dev(W8, fmt), c(s_a), ec_mode, ec, S)
    dW = s3r.int8_gemm_dw(_dev(A8, fmt), q.Q, q.tile_scale, c(s_w), ec_mode, ec, S)
    torch.cuda.synchronize()
    assert np.array_equal(codes(q.Q), ref.Q)
    mdx = dx_magnitude(ref.Q, ref.delta, W8, s_a, ref.eps, ref.rowsum, ref.v, S, rows=rows)
    assert_close_mag(dA.cpu().numpy()[rows], ref.dX, mdx, "dA rows")
    if ec_mode == orc.EC_TWO_WAY:
        mdw = dw_magnitude(A8, ref.Q, ref.delta, s_w, ref.colmean, ref.mu, ref.xsum, ref.p, krows=krows)
    else:
        mdw = dw_magnitude(A8, ref.Q, ref.delta, s_w, krows=krows)
    assert_close_mag(dW.cpu().numpy()[krows], ref.dW, mdw, "dW2 rows")
