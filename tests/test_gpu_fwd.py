"""GPU parity: the INT8 forward of the SwiGLU block.

Source: "Efficient Quantization Training with Stochastic Rounding via
Structured Subspace Randomness" -- §III-A (RTNE forward operands, per-token
and per-output-channel scales, S32 accumulation then rescale), §IV-A (the
SwiGLU FFN block; GEMM outputs kept in bf16).

Every step is integer-exact up to the fp32 roundings the oracle fixes in
order (the 128-block additions, the two rescales, the bf16 roundings and the
gate), so the comparisons are bit for bit:
1. int8_gemm_fwd against the oracle's gemm_fwd, ragged shapes included;
2. int8_gemm_fwd_swiglu against gemm_fwd + swiglu_fwd (h1, h3, a);
3. ffn_forward against ffn_forward_int8 (codes, scales, h1, h3, a, A8, Y),
   and with weights given already quantized;
4. at d = 2048, F = 5632, T = 8192 (the benchmark block), sampled rows.
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def s3r():
    import stochastic_rounding_int8_gb300 as m
    m.lib()
    return m


def _codes(rng, shape):
    return rng.integers(-127, 128, size=shape).astype(np.int8)


def _dev_codes(a):
    return torch.from_numpy(a.astype(np.float16)).cuda()


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("T,K,N", [(128, 128, 256), (300, 264, 520), (77, 1000, 136), (513, 2048, 1024),
                                   (1, 8, 8), (260, 4104, 24)])
def test_gemm_fwd_bit_exact(s3r, orc, T, K, N):
    rng = np.random.default_rng(T * 7 + K + N)
    X8, W8 = _codes(rng, (T, K)), _codes(rng, (K, N))
    s_x = (rng.random(T) * 0.05 + 1e-3).astype(np.float32)
    s_w = (rng.random(N) * 0.01 + 1e-4).astype(np.float32)
    st = s3r.new_status()
    Y = s3r.int8_gemm_fwd(_dev_codes(X8), torch.from_numpy(s_x).cuda(), _dev_codes(W8),
                          torch.from_numpy(s_w).cuda(), status=st)
    s3r.check_status(st)
    ref = orc.gemm_fwd(X8, s_x, W8, s_w)
    got = Y.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), np.abs(got - ref).max()


def test_gemm_fwd_saturated_blocks(s3r, orc):
    """All codes +-127: every block sum is at the 2^21 bound and the blocks'
    fp32 additions round; the kernel adds them in the same order."""
    T, K, N = 256, 4096, 256
    rng = np.random.default_rng(4)
    X8 = np.where(rng.random((T, K)) < 0.9, 127, -127).astype(np.int8)
    W8 = np.where(rng.random((K, N)) < 0.9, 127, -127).astype(np.int8)
    s_x = np.full(T, 0.3, np.float32)
    s_w = np.full(N, 0.7, np.float32)
    Y = s3r.int8_gemm_fwd(_dev_codes(X8), torch.from_numpy(s_x).cuda(), _dev_codes(W8), torch.from_numpy(s_w).cuda())
    ref = orc.gemm_fwd(X8, s_x, W8, s_w)
    assert np.array_equal(Y.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("T,K,F", [(256, 256, 384), (200, 136, 72), (129, 512, 1000)])
def test_gemm_fwd_swiglu_bit_exact(s3r, orc, T, K, F):
    rng = np.random.default_rng(T + K + F)
    X8, W1, W3 = _codes(rng, (T, K)), _codes(rng, (K, F)), _codes(rng, (K, F))
    s_x = (rng.random(T) * 0.02 + 1e-3).astype(np.float32)
    s_w1 = (rng.random(F) * 0.01 + 1e-4).astype(np.float32)
    s_w3 = (rng.random(F) * 0.01 + 1e-4).astype(np.float32)
    c = lambda a: torch.from_numpy(a).cuda()
    h1, h3, a = s3r.int8_gemm_fwd_swiglu(_dev_codes(X8), c(s_x), _dev_codes(W1), c(s_w1), _dev_codes(W3), c(s_w3))
    r1, r3, ra = orc.swiglu_fwd(orc.gemm_fwd(X8, s_x, W1, s_w1), orc.gemm_fwd(X8, s_x, W3, s_w3))
    assert np.array_equal(_bits(h1), r1)
    assert np.array_equal(_bits(h3), r3)
    assert np.array_equal(_bits(a), ra)


@pytest.mark.parametrize("T,F,pad", [(64, 5632, 0), (37, 8, 0), (300, 13000, 8), (5, 136, 24)])
@pytest.mark.parametrize("fmt", ["f16", "s8"])
def test_swiglu_fwd_quantize_matches_oracle(s3r, orc, T, F, pad, fmt):
    """The gate fused into the RTNE of a: a bit for bit as the oracle's
    swiglu_fwd, codes and scales as its RTNE operand of a; rows longer than
    the register-resident part recompute the gate for the codes."""
    rng = np.random.default_rng(T + F)
    std = 0.02 * np.sqrt(2048)
    full1 = torch.from_numpy((rng.standard_normal((T, F + pad)) * std).astype(np.float32)).to(torch.bfloat16)
    full3 = torch.from_numpy((rng.standard_normal((T, F + pad)) * std).astype(np.float32)).to(torch.bfloat16)
    full1[min(2, T - 1), :] = 0   # an all-zero row: a = 0, scale 1
    h1, h3 = full1[:, :F], full3[:, :F]
    cf = s3r.CODES_F16 if fmt == "f16" else s3r.CODES_S8
    a, Q, sc = s3r.swiglu_fwd_quantize(h1.cuda(), h3.cuda(), code_format=cf)
    f = lambda t: orc.bf16_to_f32(t.contiguous().view(torch.int16).numpy().view(np.uint16))
    _, _, ra = orc.swiglu_fwd(f(h1), f(h3))
    assert np.array_equal(_bits(a), ra)
    rq, rs = orc.rtne_operand(orc.bf16_to_f32(ra), 0)
    got = Q.cpu().float().numpy().astype(np.int8) if fmt == "f16" else Q.cpu().numpy()
    assert np.array_equal(got, rq)
    assert np.array_equal(sc.cpu().numpy(), rs)
    none, Q2, sc2 = s3r.swiglu_fwd_quantize(h1.cuda(), h3.cuda(), keep_a=False, code_format=cf)
    assert none is None and torch.equal(Q2, Q) and torch.equal(sc2, sc)


def test_swiglu_fwd_quantize_nonfinite_and_alignment(s3r):
    h1 = torch.randn(4, 64).to(torch.bfloat16).cuda()
    h3 = torch.randn(4, 64).to(torch.bfloat16).cuda()
    h1[1, 7] = float("inf")
    st = s3r.new_status()
    a, Q, sc = s3r.swiglu_fwd_quantize(h1, h3, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == -4   # S3R_ERR_NONFINITE
    assert torch.isnan(sc[1]).item() and torch.count_nonzero(Q[1]).item() == 0
    assert not torch.isnan(sc[[0, 2, 3]]).any()
    with pytest.raises(s3r.S3RError, match="ALIGN"):
        s3r.swiglu_fwd_quantize(h1[:, :60], h3[:, :60])


def test_gemm_fwd_pair_without_gate(s3r):
    """With a = NULL the launch writes the same h1, h3 and leaves a alone."""
    rng = np.random.default_rng(11)
    T, K, F = 192, 384, 264
    X8, W1, W3 = _codes(rng, (T, K)), _codes(rng, (K, F)), _codes(rng, (K, F))
    c = lambda a: torch.from_numpy(a).cuda()
    s_x, s_w1, s_w3 = (c((rng.random(n) * 0.01 + 1e-4).astype(np.float32)) for n in (T, F, F))
    h1, h3, a = s3r.int8_gemm_fwd_swiglu(_dev_codes(X8), s_x, _dev_codes(W1), s_w1, _dev_codes(W3), s_w3)
    g1, g3, none = s3r.int8_gemm_fwd_swiglu(_dev_codes(X8), s_x, _dev_codes(W1), s_w1, _dev_codes(W3), s_w3,
                                            with_gate=False)
    assert none is None and torch.equal(g1, h1) and torch.equal(g3, h3)


def _block(T, d, F, seed=0):
    inp = workloads.ffn_inputs(T, d, F, S=T, seed=workloads.DATA_SEED + seed)
    return inp.X, inp.W1, inp.W3, inp.W2


def _check_forward(orc, out, ref, rows=None):
    sel = slice(None) if rows is None else rows
    o = out.ops
    f16 = lambda t: t.cpu().float().numpy().astype(np.int8)
    assert np.array_equal(f16(o.X8)[sel], ref.X8)
    assert np.array_equal(o.s_x.cpu().numpy()[sel], ref.s_x)
    for got, want in ((o.W1_8, ref.W1_8), (o.W3_8, ref.W3_8), (o.W2_8, ref.W2_8)):
        assert np.array_equal(f16(got), want)
    for got, want in ((o.s_w1, ref.s_w1), (o.s_w3, ref.s_w3), (o.s_w2, ref.s_w2)):
        assert np.array_equal(got.cpu().numpy(), want)
    assert np.array_equal(_bits(o.h1)[sel], ref.h1)
    assert np.array_equal(_bits(o.h3)[sel], ref.h3)
    assert np.array_equal(_bits(out.a)[sel], ref.a)
    assert np.array_equal(f16(o.A8)[sel], ref.A8)
    assert np.array_equal(o.s_a.cpu().numpy()[sel], ref.s_a)
    got = out.Y.cpu().numpy()[sel]
    assert np.array_equal(got.view(np.uint32), ref.Y.view(np.uint32)), np.abs(got - ref.Y).max()


@pytest.mark.parametrize("T,d,F", [(256, 256, 384), (300, 136, 520)])
def test_ffn_forward_matches_oracle(s3r, orc, T, d, F):
    X, W1, W3, W2 = _block(T, d, F)
    out = s3r.ffn_forward(X.cuda(), W1.cuda(), W3.cuda(), W2.cuda())
    torch.cuda.synchronize()
    f = orc.from_torch_bf16
    ref = orc.ffn_forward_int8(f(X), f(W1), f(W3), f(W2))
    _check_forward(orc, out, ref)
    # the same block with the weights handed in already quantized
    again = s3r.alloc_ffn_forward(T, d, F)
    for name in ("W1_8", "s_w1", "W3_8", "s_w3", "W2_8", "s_w2"):
        getattr(again.ops, name).copy_(getattr(out.ops, name))
    s3r.ffn_forward(X.cuda(), out=again, quantize_weights=False)
    assert torch.equal(again.Y, out.Y) and torch.equal(again.a, out.a)
    # without keeping a (the backward reads only its codes)
    lean = s3r.ffn_forward(X.cuda(), W1.cuda(), W3.cuda(), W2.cuda(), keep_a=False)
    assert lean.a is None and torch.equal(lean.Y, out.Y) and torch.equal(lean.ops.A8, out.ops.A8)


def test_ffn_forward_full_size_sampled_rows(s3r, orc):
    """The benchmark block (T = 8192, d = 2048, F = 5632): the oracle's
    forward of 24 sampled tokens (rows are independent in the forward)."""
    T, d, F = 8192, 2048, 5632
    X, W1, W3, W2 = _block(T, d, F, seed=3)
    st = s3r.new_status()
    out = s3r.ffn_forward(X.cuda(), W1.cuda(), W3.cuda(), W2.cuda(), status=st)
    s3r.check_status(st)
    rows = np.sort(np.random.default_rng(5).choice(T, 24, replace=False))
    rows[0], rows[-1] = 0, T - 1
    f = orc.from_torch_bf16
    ref = orc.ffn_forward_int8(f(X[torch.from_numpy(rows)]), f(W1), f(W3), f(W2))
    _check_forward(orc, out, ref, rows)


def test_forward_edge_cases(s3r):
    dev = "cuda"
    X8 = torch.ones((4, 0), dtype=torch.float16, device=dev)
    W8 = torch.ones((0, 16), dtype=torch.float16, device=dev)
    s = torch.ones(16, device=dev)
    Y = torch.full((4, 16), 7.0, device=dev)
    s3r.int8_gemm_fwd(X8, s[:4], W8, s, Y=Y)
    assert torch.count_nonzero(Y).item() == 0
    h1, h3, a = s3r.int8_gemm_fwd_swiglu(X8, s[:4], W8, s, W8, s)
    assert all(torch.count_nonzero(t).item() == 0 for t in (h1, h3, a))
    # empty token dimension: nothing to do
    s3r.int8_gemm_fwd(torch.ones((0, 16), dtype=torch.float16, device=dev), s[:0],
                      torch.ones((16, 16), dtype=torch.float16, device=dev), s)
    # N not a multiple of 8: 16-byte rows are required
    with pytest.raises(s3r.S3RError, match="ALIGN"):
        s3r.int8_gemm_fwd(torch.ones((8, 16), dtype=torch.float16, device=dev), s[:8],
                          torch.ones((16, 12), dtype=torch.float16, device=dev), s[:12])
    # int8-carried codes are not taken by the forward
    with pytest.raises(s3r.S3RError, match="UNSUPPORTED"):
        s3r.int8_gemm_fwd(torch.ones((8, 16), dtype=torch.int8, device=dev), s[:8],
                          torch.ones((16, 16), dtype=torch.int8, device=dev), s)


@pytest.mark.parametrize("R,C,pad", [(300, 264, 0), (77, 13000, 8), (2048, 5632, 0), (5632, 2048, 0), (33, 12, 0),
                                     (19, 100, 3), (600, 8, 0)])
@pytest.mark.parametrize("fmt", ["f16", "s8"])
def test_rtne_operand_row_and_column_scales(s3r, orc, R, C, pad, fmt):
    """rtne_quantize per row and per column against the oracle's RTNE operand:
    16-byte rows (vector kernels, rows longer than the register-resident
    part included) and odd widths or strides (element kernels); an all-zero
    row and column, and a row and a column holding an Inf."""
    rng = np.random.default_rng(R + C + pad)
    full = torch.from_numpy((rng.standard_normal((R, C + pad)) * 0.02).astype(np.float32)).to(torch.bfloat16)
    full[1, :] = 0
    full[:, 2] = 0
    A = full[:, :C]
    cf = s3r.CODES_F16 if fmt == "f16" else s3r.CODES_S8
    f = lambda t: orc.bf16_to_f32(t.contiguous().view(torch.int16).numpy().view(np.uint16))
    for axis in (s3r.AXIS_ROW, s3r.AXIS_COL):
        Q, sc = s3r.rtne_quantize(A.cuda(), axis, code_format=cf)
        rq, rs = orc.rtne_operand(f(A), 0 if axis == s3r.AXIS_ROW else 1)
        got = Q.cpu().float().numpy().astype(np.int8) if fmt == "f16" else Q.cpu().numpy()
        assert np.array_equal(got, rq)
        assert np.array_equal(sc.cpu().numpy(), rs)
    # a non-finite value: its row (column) codes to 0 with a NaN scale and the status flag
    B = A.clone()
    B[3, 5] = float("inf")
    for axis, idx in ((s3r.AXIS_ROW, 3), (s3r.AXIS_COL, 5)):
        st = s3r.new_status()
        Q, sc = s3r.rtne_quantize(B.cuda(), axis, code_format=cf, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == -4   # S3R_ERR_NONFINITE
        q = Q.cpu().float()
        line = q[idx] if axis == s3r.AXIS_ROW else q[:, idx]
        assert torch.count_nonzero(line).item() == 0 and torch.isnan(sc[idx]).item()
        clean = torch.ones(sc.numel(), dtype=torch.bool)
        clean[idx] = False
        ref_q, ref_s = s3r.rtne_quantize(A.cuda(), axis, code_format=cf)
        assert torch.equal(sc.cpu()[clean], ref_s.cpu()[clean])
        keep = (q != ref_q.cpu().float())
        if axis == s3r.AXIS_ROW:
            keep[idx] = False
        else:
            keep[:, idx] = False
        assert not keep.any()
