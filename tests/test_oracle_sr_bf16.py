"""Pins for the oracle's stochastic rounding of fp32 to bf16 with shared
16-bit thresholds.

Source: "Efficient Quantization Training with Stochastic Rounding via
Structured Subspace Randomness" -- §II (hardware SR to floating-point formats
from program-supplied random bits), §III-B (one threshold per token);
"Stochastic Rounding" (transformer-math blog) -- "Stochastic rounding,
defined", "The probability formula", "A worked example: the weight RTN
freezes".
"""
import json
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sr_worked_example.json")


def _neighbours(x):
    """The two bf16 values around fp32 x (toward zero, away from zero), from
    the torch round-toward-zero of the magnitude in float64."""
    x = np.float32(x)
    mag = abs(float(x))
    lo = np.float32(mag).view(np.uint32) & np.uint32(0xFFFF0000)
    lo_v = float(lo.view(np.float32))
    hi_v = float((lo + np.uint32(0x10000)).view(np.float32))
    return lo_v, hi_v


def test_probability_is_distance_over_spacing(orc):
    """The magnitude rounds up exactly for the thresholds v < c, where
    c / 2^16 = (|x| - lo) / (hi - lo) is computed from the two bf16
    neighbours in float64: so over uniform 16-bit thresholds the probability
    of rounding up is the distance to the lower neighbour over the spacing."""
    rng = np.random.default_rng(1)
    xs = (rng.standard_normal(400) * 10.0 ** rng.integers(-30, 30, 400)).astype(np.float32)
    for x in xs:
        lo, hi = _neighbours(x)
        c = (abs(float(x)) - lo) / (hi - lo) * 65536
        assert c == int(c)
        c = int(c)
        lo_bits = int(np.float32(lo).view(np.uint32) >> 16)
        up = lambda v: (orc.sr_bf16_scalar(float(x), v) & 0x7FFF) != lo_bits
        if c > 0:
            assert up(0) and up(c - 1)
        assert not up(c) and not up(65535)


def test_on_grid_values_never_move_and_sign_is_kept(orc):
    rng = np.random.default_rng(2)
    grid = torch.from_numpy(rng.standard_normal(200).astype(np.float32)).to(torch.bfloat16)
    bits = grid.view(torch.int16).numpy().view(np.uint16)
    vals = grid.float().numpy()
    for b, x in zip(bits, vals):
        for v in (0, 1, 30000, 65535):
            assert orc.sr_bf16_scalar(float(x), v) == int(b)
    assert orc.sr_bf16_scalar(-1.00390625 - 2 ** -10, 0) & 0x8000


def test_worked_example_mean_and_rtn_freeze(orc):
    """[SRB]'s 256.3: in bf16 the neighbours are 256 and 258, RTN gives 256
    every time (the update freezes) and SR lands on 258 with probability
    0.15; the mean over independent thresholds is 256.3 within 3 sigma."""
    ex = json.load(open(GOLDEN))
    x = float(np.float32(ex["x"]))
    assert orc.bf16_to_f32(np.array([orc.to_bf16_bits(np.array([x], np.float32))[0]]))[0] == 256.0
    rng = np.random.default_rng(3)
    vs = rng.integers(0, 65536, size=20000)
    out = orc.bf16_to_f32(np.array([orc.sr_bf16_scalar(x, int(v)) for v in vs], dtype=np.uint16))
    assert set(np.unique(out)) <= {256.0, 258.0}
    p = (x - 256.0) / 2.0
    sigma = 2.0 * np.sqrt(p * (1 - p) / len(vs))
    assert abs(out.mean() - x) <= 3 * sigma


def test_matrix_s3r_shares_one_threshold_per_token(orc):
    """Within a token, rounding up is monotone in the dropped bits and its
    cut equals the token's Philox word (upper 16 bits); INDEP draws per
    element from word e mod 4 of Philox(e / 4)."""
    rng = np.random.default_rng(4)
    T, N = 24, 300
    X = (rng.standard_normal((T, N)) * 3).astype(np.float32)
    Y = orc.sr_bf16(X, orc.S3R, seed=7, tensor_id=5)
    lows = X.view(np.uint32) & 0xFFFF
    up = (Y & 0x7FFF) != ((np.abs(X).view(np.uint32) >> 16) & 0x7FFF)
    for t in range(T):
        v = int(orc.philox4x32_10([t, 0, 0, 0], [7, 5])[0]) >> 16
        assert np.array_equal(up[t], lows[t] > v)
    # a window of rows starting at token 10 equals those rows of the whole
    assert np.array_equal(orc.sr_bf16(X[10:14], orc.S3R, seed=7, tensor_id=5, t0=10), Y[10:14])
    assert np.array_equal(orc.sr_bf16(X[10:14], orc.INDEP, seed=7, tensor_id=5, t0=10),
                          orc.sr_bf16(X, orc.INDEP, seed=7, tensor_id=5)[10:14])
    Yi = orc.sr_bf16(X, orc.INDEP, seed=7, tensor_id=5)
    upi = (Yi & 0x7FFF) != ((np.abs(X).view(np.uint32) >> 16) & 0x7FFF)
    for t in (0, 5, 23):
        for n in (0, 1, 2, 3, 299):
            e = t * N + n
            v = int(orc.philox4x32_10([e // 4, 0, 0, 0], [7, 5])[e % 4]) >> 16
            assert upi[t, n] == (lows[t, n] > v)


def test_matrix_unbiased_over_seeds(orc):
    rng = np.random.default_rng(6)
    X = (rng.standard_normal((4, 64)) * 5).astype(np.float32)
    acc = np.zeros(X.shape)
    seeds = 1500
    for sd in range(seeds):
        acc += orc.bf16_to_f32(orc.sr_bf16(X, orc.S3R, seed=sd, tensor_id=1))
    spacing = np.abs(X) * 2.0 ** -7
    assert np.all(np.abs(acc / seeds - X) <= 5 * 0.5 * spacing / np.sqrt(seeds) + 1e-12)


def test_rtne_and_saturation(orc):
    rng = np.random.default_rng(7)
    X = (rng.standard_normal((8, 50)) * 100).astype(np.float32)
    ref = torch.from_numpy(X).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.sr_bf16(X, orc.RTNE), ref)
    big = np.array([[3.4e38, -np.inf, np.inf, np.nan]], dtype=np.float32)
    Y = orc.sr_bf16(big, orc.S3R, seed=1)
    assert Y[0, 0] == 0x7F7F and Y[0, 1] == 0xFF7F and Y[0, 2] == 0x7F7F and Y[0, 3] == 0x7FFF
