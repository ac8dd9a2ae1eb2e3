"""GPU parity: stochastic rounding of fp32 to bf16, and to FP8 e4m3 after a
scale, with S3R's shared thresholds on the hardware conversions.

Source: "Efficient Quantization Training with Stochastic Rounding via
Structured Subspace Randomness" -- §II (hardware SR to floating-point formats
from supplied random bits), §III-B (one threshold per token).

The rounding is a bit operation on the fp32 pattern, so the comparison with
the oracle is bit for bit: vector and element paths, ragged widths, strides,
all three modes, saturation, and sampled rows at [16384, 8192].
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


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


_MODES = {"s3r": ("ROUND_S3R", "S3R"), "indep": ("ROUND_INDEP", "INDEP"), "rtne": ("ROUND_RTNE", "RTNE")}


@pytest.mark.parametrize("T,N,pad", [(64, 8192, 0), (33, 8200, 0), (17, 1000, 4), (9, 77, 3), (300, 24, 0),
                                     (3, 16385, 1)])
@pytest.mark.parametrize("mode", ["s3r", "indep", "rtne"])
def test_sr_bf16_matches_oracle(s3r, orc, T, N, pad, mode):
    rng = np.random.default_rng(T * 31 + N + pad)
    full = (rng.standard_t(3, size=(T, N + pad)) * 10.0 ** rng.integers(-4, 4, (T, 1))).astype(np.float32)
    X = full[:, :N]
    sm, om = _MODES[mode]
    Xd = torch.from_numpy(full).cuda()[:, :N]
    Y = s3r.s3r_sr_bf16(Xd, getattr(s3r, sm), seed=11, tensor_id=3)
    ref = orc.sr_bf16(np.ascontiguousarray(X), getattr(orc, om), seed=11, tensor_id=3)
    assert np.array_equal(_bits(Y), ref)


def test_sr_bf16_strided_output_and_saturation(s3r, orc):
    X = np.array([[3.4e38, -3.4e38, np.inf, -np.inf, 1.0, -2.5, 1e-40, 0.0]] * 4, dtype=np.float32)
    Yfull = torch.zeros((4, 16), dtype=torch.bfloat16, device="cuda")
    s3r.s3r_sr_bf16(torch.from_numpy(X).cuda(), s3r.ROUND_S3R, seed=2, Y=Yfull[:, 3:11])
    got = _bits(Yfull)
    assert np.array_equal(got[:, 3:11], orc.sr_bf16(X, orc.S3R, seed=2))
    assert not got[:, :3].any() and not got[:, 11:].any()
    assert got[0, 3] == 0x7F7F and got[0, 4] == 0xFF7F and got[0, 5] == 0x7F7F and got[0, 6] == 0xFF7F
    nan = torch.full((1, 8), float("nan"), device="cuda")
    out = s3r.s3r_sr_bf16(nan, s3r.ROUND_S3R)
    assert torch.isnan(out.float()).all()


def test_sr_bf16_full_size_sampled_rows(s3r, orc):
    """[16384, 8192] fp32 (the sweep size): sampled rows equal the oracle."""
    T, N = 16384, 8192
    G = workloads.quantize_sweep_input(T, N, seed=workloads.DATA_SEED + 3).float() * 1e3
    Y = s3r.s3r_sr_bf16(G.cuda(), s3r.ROUND_S3R, seed=5, tensor_id=1)
    rows = np.sort(np.random.default_rng(9).choice(T, 12, replace=False))
    rows[-1] = T - 1
    Xr = G.numpy()[rows]
    got = _bits(Y)[rows]
    for i, t in enumerate(rows):
        ref = orc.sr_bf16(np.ascontiguousarray(Xr[i:i + 1]), orc.S3R, seed=5, tensor_id=1, t0=int(t))
        assert np.array_equal(got[i:i + 1], ref)


def test_sr_bf16_rejects_bad_arguments(s3r):
    X = torch.ones((4, 8), device="cuda")
    with pytest.raises(s3r.S3RError, match="ARG"):
        s3r.s3r_sr_bf16(X, s3r.ROUND_S3R_7BIT)
    with pytest.raises(AssertionError):
        s3r.s3r_sr_bf16(X.to(torch.bfloat16))


# --- FP8 e4m3 ------------------------------------------------------------
@pytest.mark.parametrize("T,N,pad", [(64, 8192, 0), (33, 8200, 0), (17, 1000, 4), (9, 77, 3), (3, 16385, 1)])
@pytest.mark.parametrize("mode", ["s3r", "indep", "rtne"])
@pytest.mark.parametrize("inv", [1.0, 0.37])
def test_sr_fp8_matches_oracle(s3r, orc, T, N, pad, mode, inv):
    """y = x * inv_scale, then e4m3 codes bit for bit: vector and element
    paths, ragged widths and strides, subnormal to saturated magnitudes."""
    rng = np.random.default_rng(T * 13 + N + pad)
    mag = 10.0 ** rng.uniform(-4.0, 3.0, size=(T, N + pad))
    full = (np.sign(rng.standard_normal((T, N + pad))) * mag).astype(np.float32)
    X = full[:, :N]
    sm, om = _MODES[mode]
    Y = s3r.s3r_sr_fp8(torch.from_numpy(full).cuda()[:, :N], inv, getattr(s3r, sm), seed=3, tensor_id=9)
    ref = orc.sr_fp8(np.ascontiguousarray(X), inv, getattr(orc, om), seed=3, tensor_id=9)
    assert np.array_equal(Y.cpu().numpy(), ref)


def test_sr_fp8_special_values_and_full_size_rows(s3r, orc):
    X = np.array([[448.0, -448.0, 1e9, -np.inf, np.inf, 0.0, -0.0, 2.0 ** -12]] * 2, dtype=np.float32)
    Y = s3r.s3r_sr_fp8(torch.from_numpy(X).cuda(), 1.0, s3r.ROUND_S3R, seed=1).cpu().numpy()
    assert np.array_equal(Y, orc.sr_fp8(X, 1.0, orc.S3R, seed=1))
    assert list(Y[0, :5]) == [0x7E, 0xFE, 0x7E, 0xFE, 0x7E]
    nan = s3r.s3r_sr_fp8(torch.full((1, 8), float("nan"), device="cuda"))
    assert torch.all((nan & 0x7F) == 0x7F)
    # [16384, 8192] at the sweep size: sampled rows equal the oracle's window
    T, N = 16384, 8192
    G = workloads.quantize_sweep_input(T, N, seed=workloads.DATA_SEED + 3).float() * 1e3
    Yf = s3r.s3r_sr_fp8(G.cuda(), 2.0, s3r.ROUND_S3R, seed=5, tensor_id=1).cpu().numpy()
    for t in (0, 4097, T - 1):
        ref = orc.sr_fp8(np.ascontiguousarray(G.numpy()[t:t + 1]), 2.0, orc.S3R, seed=5, tensor_id=1, t0=t)
        assert np.array_equal(Yf[t:t + 1], ref)
