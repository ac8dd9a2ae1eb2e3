"""GPU parity: stochastic rounding of fp32 to bf16 with S3R's shared
thresholds on the hardware conversion.

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
