"""Pins for the oracle's stochastic rounding of fp32 to FP8 e4m3 with shared
16-bit thresholds.

Source: "Efficient Quantization Training with Stochastic Rounding via
Structured Subspace Randomness" -- §II (hardware SR to floating-point formats
from program-supplied random bits), §III-B (one threshold per token);
"Stochastic Rounding" (transformer-math blog) -- "The probability formula".
The e4m3 grid itself comes from torch's float8_e4m3fn type (a library
definition independent of the oracle).
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.skipif(not hasattr(torch, "float8_e4m3fn"), reason="torch without float8_e4m3fn")


def _grid():
    """All non-negative finite e4m3 values (codes 0x00 .. 0x7E), from torch."""
    codes = torch.arange(0, 0x7F, dtype=torch.uint8)
    return codes.view(torch.float8_e4m3fn).float().numpy().astype(np.float64)


def _decode(codes):
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).float().numpy()


def test_grid_codes_never_move(orc):
    g = _grid()
    for code, val in enumerate(g):
        for v in (0, 1, 40000, 65535):
            assert orc.sr_e4m3_scalar(val, v) == code
            assert orc.sr_e4m3_scalar(-val, v) == (code | 0x80)
        assert orc.rn_e4m3_scalar(val) == code


def test_cut_at_the_probability_formula(orc):
    """Between grid neighbours lo < |y| < hi the magnitude rounds up exactly
    for v < c with c = floor(2^16 (|y| - lo) / (hi - lo)) (float64, torch grid)."""
    g = _grid()
    rng = np.random.default_rng(1)
    ys = (rng.random(600) * 447.0 * np.exp(-rng.random(600) * 20)).astype(np.float32)
    for y in ys:
        m = float(y)
        i = np.searchsorted(g, m, side="right") - 1
        lo, hi = g[i], g[i + 1]
        if m == lo:
            continue
        c = int(np.floor((m - lo) / (hi - lo) * 65536.0))
        up = lambda v: _decode([orc.sr_e4m3_scalar(m, v)])[0] == hi
        dn = lambda v: _decode([orc.sr_e4m3_scalar(m, v)])[0] == lo
        if c > 0:
            assert up(0) and up(c - 1)
        assert dn(c) and dn(65535)


def test_rtne_equals_torch_and_saturation(orc):
    rng = np.random.default_rng(2)
    y = (rng.standard_normal(3000) * 10.0 ** rng.integers(-3, 3, 3000)).astype(np.float32)
    y = y[np.abs(y) < 440]
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.rn_e4m3_scalar(float(v)) for v in y], dtype=np.uint8)
    assert np.array_equal(got, ref)
    for v, want in ((448.0, 0x7E), (1e9, 0x7E), (-1e9, 0xFE), (float("inf"), 0x7E), (-float("inf"), 0xFE),
                    (450.0, 0x7E)):
        assert orc.sr_e4m3_scalar(v, 0) == want and orc.rn_e4m3_scalar(v) == want
    assert orc.sr_e4m3_scalar(float("nan"), 0) == 0x7F


def test_matrix_modes_window_scale_and_sharing(orc):
    rng = np.random.default_rng(3)
    T, N = 20, 96
    X = (rng.standard_normal((T, N)) * 30).astype(np.float32)
    Y = orc.sr_fp8(X, 0.5, orc.S3R, seed=7, tensor_id=4)
    # the scale is one fp32 multiply before the rounding
    assert np.array_equal(Y, orc.sr_fp8((X * np.float32(0.5)).astype(np.float32), 1.0, orc.S3R, seed=7, tensor_id=4))
    # windows equal slices
    assert np.array_equal(orc.sr_fp8(X[5:9], 0.5, orc.S3R, seed=7, tensor_id=4, t0=5), Y[5:9])
    assert np.array_equal(orc.sr_fp8(X[5:9], 0.5, orc.INDEP, seed=7, tensor_id=4, t0=5),
                          orc.sr_fp8(X, 0.5, orc.INDEP, seed=7, tensor_id=4)[5:9])
    # S3R: per token the cut is the token word's upper 16 bits
    g = _grid()
    for t in range(T):
        v = int(orc.philox4x32_10([t, 0, 0, 0], [7, 4])[0]) >> 16
        for n in range(N):
            m = abs(float(np.float32(X[t, n] * np.float32(0.5))))
            if m >= 448:
                continue
            i = np.searchsorted(g, m, side="right") - 1
            lo, hi = g[i], g[i + 1]
            c = int(np.floor((m - lo) / (hi - lo) * 65536.0))
            assert abs(_decode([Y[t, n]])[0]) == (hi if c > v else lo)


def test_unbiased_over_seeds(orc):
    rng = np.random.default_rng(4)
    X = (rng.standard_normal((4, 32)) * 20).astype(np.float32)
    acc = np.zeros(X.shape)
    seeds = 1500
    for sd in range(seeds):
        acc += _decode(orc.sr_fp8(X, 1.0, orc.S3R, seed=sd, tensor_id=2)).astype(np.float64)
    spacing = np.maximum(2.0 ** (np.floor(np.log2(np.abs(X))) - 3), 2.0 ** -9)
    assert np.all(np.abs(acc / seeds - X) <= 5 * 0.5 * spacing / np.sqrt(seeds) + spacing * 2.0 ** -16)
