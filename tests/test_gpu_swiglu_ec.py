"""GPU parity: the SwiGLU-fused quantizer and the S3R-EC correction factors."""
import numpy as np
import pytest
import torch

from parity_util import assert_close_mag, codes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def s3r():
    import stochastic_rounding_int8_gb300 as m
    m.lib()
    return m


def _swiglu_case(T, F, seed):
    rng = np.random.default_rng(seed)
    dA = (rng.standard_normal((T, F)) * 3e-4).astype(np.float32)
    h1 = torch.from_numpy((rng.standard_normal((T, F)) * 0.9).astype(np.float32)).to(torch.bfloat16)
    h3 = torch.from_numpy((rng.standard_normal((T, F)) * 0.9).astype(np.float32)).to(torch.bfloat16)
    s_x = (rng.random(T) * 0.03 + 0.02).astype(np.float32)
    s_w1 = (rng.random(F) * 5e-4 + 1e-4).astype(np.float32)
    s_w3 = (rng.random(F) * 5e-4 + 1e-4).astype(np.float32)
    return dA, h1, h3, s_x, s_w1, s_w3


@pytest.mark.parametrize("fmt", [0, 1], ids=["s8", "f16"])
@pytest.mark.parametrize("mode", ["S3R", "INDEP", "RTNE", "S3R_7BIT", "BCAST"])
@pytest.mark.parametrize("T,F", [(256, 384), (300, 200), (129, 1000), (64, 8)])
def test_swiglu_quantize_parity(s3r, orc, fmt, mode, T, F):
    dA, h1, h3, s_x, s_w1, s_w3 = _swiglu_case(T, F, T + F)
    S = 128 if mode == "BCAST" and T % 128 == 0 else 0
    c = lambda a: torch.from_numpy(a).cuda()
    o1, o3 = s3r.swiglu_quantize(c(dA), h1.cuda(), h3.cuda(), c(s_x), c(s_w1), c(s_w3),
                                 round_mode=getattr(s3r, "ROUND_" + mode), seed=42, tid1=1, tid3=2, code_format=fmt,
                                 S=S)
    torch.cuda.synchronize()
    dh1, dh3 = orc.swiglu_bwd(dA, orc.from_torch_bf16(h1), orc.from_torch_bf16(h3))
    omode = orc.S3R7 if mode == "S3R_7BIT" else getattr(orc, mode)
    for o, g, s_w, tid in ((o1, dh1, s_w1, 1), (o3, dh3, s_w3, 2)):
        Qo, do, Eo, st = orc.quantize(g, s_x, s_w, mode=omode, seed=42, tensor_id=tid, S=S)
        assert st == 0
        Qg = codes(o.Q)
        assert np.array_equal(Qg, Qo), f"{mode} tid {tid}: {(Qg != Qo).sum()} codes differ"
        assert np.array_equal(o.tile_scale.cpu().numpy(), do)
        if omode in orc.SHARED:
            t_o, c_o = orc.error_partials(Eo)
            t_m, c_m = orc.error_partials(np.abs(Eo))
            assert_close_mag(o.tok_err_part.cpu().numpy(), t_o, t_m, "tok")
            assert_close_mag(o.col_err_part.cpu().numpy(), c_o, c_m, "col")


@pytest.mark.parametrize("fmt", [0, 1], ids=["s8", "f16"])
@pytest.mark.parametrize("ec_mode", ["EC_DX_ONLY", "EC_TWO_WAY", "EC_DW_ONLY"])
@pytest.mark.parametrize("T,N,K,S", [(256, 1024, 512, 256), (512, 384, 200, 128), (300, 260, 72, 300),
                                     (1024, 256, 130, 256), (1280, 256, 136, 128), (384, 5632, 264, 128),
                                     (512, 7000, 264, 128), (256, 512, 5008, 128)])
def test_ec_factors_parity(s3r, orc, fmt, ec_mode, T, N, K, S):
    rng = np.random.default_rng(T + N + K)
    G = (rng.standard_t(3, size=(T, N)) * 1e-3).astype(np.float32)
    Gb = torch.from_numpy(G).to(torch.bfloat16)
    W8 = rng.integers(-127, 128, size=(K, N)).astype(np.int8)
    X8 = rng.integers(-127, 128, size=(T, K)).astype(np.int8)
    dt = torch.float16 if fmt else torch.int8
    q = s3r.s3r_quantize(Gb.cuda(), seed=3, tensor_id=9, code_format=fmt)
    ec = s3r.s3r_ec_correct(q, T, N, S, torch.from_numpy(W8).to(dt).cuda(), torch.from_numpy(X8).to(dt).cuda(),
                            ec_mode=getattr(s3r, ec_mode))
    torch.cuda.synchronize()
    Qo, do, Eo, _ = orc.quantize(orc.from_torch_bf16(Gb), seed=3, tensor_id=9)
    eps, colmean, mu = orc.error_stats(Eo, S)
    rowsum, v, xsum, p = orc.ec_factors(eps, colmean, mu, S, W8, X8)
    B = T // S
    absE = np.abs(Eo).astype(np.float64)
    eps_m = absE.sum(1) / N
    cm_m = absE.reshape(B, S, N).sum(1) / S
    mu_m = absE.reshape(B, -1).sum(1) / (S * N)
    assert_close_mag(ec.eps.cpu().numpy(), eps, eps_m, "eps")
    assert_close_mag(ec.colmean.cpu().numpy(), colmean, cm_m, "colmean")
    assert_close_mag(ec.mu.cpu().numpy(), mu, mu_m, "mu")
    if ec_mode != "EC_DW_ONLY":   # the weight-side factors are not needed by the dW-only ablation
        assert np.array_equal(ec.rowsum.cpu().numpy(), rowsum)
        v_m = (np.abs(colmean) + np.abs(mu)[:, None]) @ np.abs(W8.astype(np.float64)).T
        assert_close_mag(ec.v.cpu().numpy(), v, v_m + cm_m @ np.abs(W8.astype(np.float64)).T, "v")
    if ec_mode in ("EC_TWO_WAY", "EC_DW_ONLY"):
        assert np.array_equal(ec.xsum.cpu().numpy(), xsum)
        p_m = np.abs(X8.astype(np.float64)).T @ (np.abs(eps) + eps_m)
        assert_close_mag(ec.p.cpu().numpy(), p, p_m, "p")


@pytest.mark.parametrize("fmt", [0, 1], ids=["s8", "f16"])
def test_ec_factors_repeat_bit_identical(s3r, fmt):
    """Two calls in a row (the column-sum pass keeps per-column-block counters
    in the workspace) give the same bits, and so does a fresh workspace."""
    rng = np.random.default_rng(5)
    T, N, K, S = 1024, 512, 264, 256
    G = torch.from_numpy((rng.standard_t(3, size=(T, N)) * 1e-3).astype(np.float32)).to(torch.bfloat16).cuda()
    dt = torch.float16 if fmt else torch.int8
    W8 = torch.from_numpy(rng.integers(-127, 128, size=(K, N)).astype(np.int8)).to(dt).cuda()
    X8 = torch.from_numpy(rng.integers(-127, 128, size=(T, K)).astype(np.int8)).to(dt).cuda()
    q = s3r.s3r_quantize(G, seed=1, tensor_id=3, code_format=fmt)
    runs = [s3r.s3r_ec_correct(q, T, N, S, W8, X8, ec_mode=s3r.EC_TWO_WAY) for _ in range(3)]
    torch.cuda.synchronize()
    for r in runs[1:]:
        for f in ("eps", "mu", "colmean", "rowsum", "v", "xsum", "p"):
            assert torch.equal(getattr(r, f), getattr(runs[0], f)), f


def test_streaming_paths_are_taken(s3r):
    """With fp16 codes and 16-byte aligned rows the quantizers run as one
    persistent launch each and the correction factors as two (the means, then
    one pass over W8 and X8); the counter sees every kernel the library starts."""
    rng = np.random.default_rng(11)
    T, N, K, S = 1024, 512, 264, 256
    G = torch.from_numpy((rng.standard_t(3, size=(T, N)) * 1e-3).astype(np.float32)).to(torch.bfloat16).cuda()
    W8 = torch.from_numpy(rng.integers(-127, 128, size=(K, N)).astype(np.float16)).cuda()
    X8 = torch.from_numpy(rng.integers(-127, 128, size=(T, K)).astype(np.float16)).cuda()
    n0 = s3r.kernel_launch_count()
    q = s3r.s3r_quantize(G, seed=1, tensor_id=3, code_format=s3r.CODES_F16)
    n1 = s3r.kernel_launch_count()
    s3r.s3r_ec_correct(q, T, N, S, W8, X8, ec_mode=s3r.EC_TWO_WAY)
    n2 = s3r.kernel_launch_count()
    s3r.s3r_ec_correct(q, T, N, S, W8, X8, ec_mode=s3r.EC_DX_ONLY)
    n3 = s3r.kernel_launch_count()
    dA, h1, h3, s_x, s_w1, s_w3 = _swiglu_case(256, 384, 2)
    c = lambda a: torch.from_numpy(a).cuda()
    s3r.swiglu_quantize(c(dA), h1.cuda(), h3.cuda(), c(s_x), c(s_w1), c(s_w3), code_format=s3r.CODES_F16)
    n4 = s3r.kernel_launch_count()
    torch.cuda.synchronize()
    assert (n1 - n0, n2 - n1, n3 - n2, n4 - n3) == (1, 2, 2, 1)


def test_glue_reciprocal_equals_ieee_everywhere(s3r):
    """sigma = 1 / (1 + e) in the glue ([S3R] section IV-A's SwiGLU block) uses
    the hardware reciprocal approximation refined by one Newton-Raphson step,
    with the IEEE reciprocal for results below the normal range.  1 + e lies in
    [1, 1 + e^88], so every float from 1.0 to the largest finite one is checked
    against the correctly rounded reciprocal: no difference anywhere."""
    one, two126, top = 0x3F800000, 0x7E800000, 0x7F800000
    assert s3r.check_reciprocal(one, two126) == 0
    assert s3r.check_reciprocal(two126, top) == 0
