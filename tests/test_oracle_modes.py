"""Pins for the oracle's paper-faithful quantizer modes and the dW-only ablation.

Source: "Efficient Quantization Training with Stochastic Rounding via
Structured Subspace Randomness" -- §III-B (7-bit thresholds, four per 32-bit
word, on a grid shifted by half a step, rounding bias at most Delta/256;
Phi_bcast: one threshold per example), §III-A (per-tensor step
max|G'|/127), Table II (the dW-only correction row).
"""
import numpy as np
import pytest


def _grid_case(rows, n, y0, p, rng):
    """A tile whose every element sits at y = y0 + p on the code grid (Delta = 1)."""
    G = np.full((rows, n), np.float32(y0 + p), dtype=np.float32)
    G[0, 0] = np.float32(127.0)          # amax = 127: Delta = 1 and inv = 1 exactly
    return G


def test_7bit_thresholds_lie_on_the_shifted_grid_and_are_uniform(orc):
    """u takes only the values (2k + 1)/256, k = 0..127, each about equally often."""
    us = np.array([orc.token_threshold7(t, 5, 3) for t in range(128 * 200)], dtype=np.float64)
    k = us * 256.0
    assert np.all(np.abs(k - np.round(k)) < 1e-9) and np.all(np.round(k) % 2 == 1)
    counts = np.bincount(((np.round(k) - 1) // 2).astype(int), minlength=128)
    assert counts.size == 128
    expected = us.size / 128
    chi2 = ((counts - expected) ** 2 / expected).sum()
    assert chi2 < 127 + 6 * np.sqrt(2 * 127)      # 127 degrees of freedom, ~6 sigma


def test_7bit_four_thresholds_per_word(orc):
    """Tokens 4w .. 4w + 3 draw from one word: the four bytes of a word are
    cut from one 32-bit value, so their concatenated upper 7 bits reproduce
    the upper 7 bits of each byte of the tokens' shared Philox word 0."""
    seed, tid = 11, 7
    for w in range(64):
        word = int(orc.philox4x32_10([w, 0, 0, 0], [seed, tid])[0])
        for i in range(4):
            k = (word >> (8 * i + 1)) & 0x7F
            assert orc.token_threshold7(4 * w + i, seed, tid) == pytest.approx((k + 0.5) / 128, abs=0)


@pytest.mark.parametrize("p", [0.0, 1 / 512, 0.1, 0.25, 0.5, 0.7, 0.999])
def test_7bit_bias_bounded_by_delta_over_256(orc, p):
    """Over many tokens (independent 7-bit thresholds) the mean code exceeds
    y by at most Delta/256 plus sampling noise, and a value on the grid
    (p = 0) never moves."""
    rng = np.random.default_rng(0)
    rows, n = 128 * 64, 8
    G = _grid_case(rows, n, 3.0, p, rng)
    Q, delta, _, st = orc.quantize(G, mode=orc.S3R7, seed=2, tensor_id=1, tile=(rows, n))
    assert st == 0 and delta[0, 0] == np.float32(1.0)
    q = Q[1:, 0].astype(np.float64)            # one element per token (column 0 of each row but the first)
    y = float(np.float32(3.0 + p))
    frac = y - 3.0
    exact_up = np.ceil(128 * frac - 0.5) / 128 if frac > 0 else 0.0   # P(u < p) on the shifted grid
    assert abs(exact_up - frac) <= 1 / 256 + 1e-12
    sigma = np.sqrt(max(exact_up * (1 - exact_up), 1e-12) / q.size)
    assert abs(q.mean() - (3.0 + exact_up)) <= 4 * sigma + 1e-12
    assert abs(q.mean() - y) <= 1 / 256 + 4 * sigma + 1e-12
    if p == 0.0:
        assert np.all(Q[1:] == 3)


def test_7bit_same_direction_per_token(orc):
    rng = np.random.default_rng(3)
    G = (rng.standard_normal((256, 384)) * 1e-2).astype(np.float32)
    Q, _, _, _ = orc.quantize(G, mode=orc.S3R7, seed=4, tensor_id=2)
    for t in range(256):
        u = orc.token_threshold7(t, 4, 2)
        for j in range(3):
            amax = np.abs(G[128 * (t // 128):128 * (t // 128 + 1), 128 * j:128 * (j + 1)]).max()
            inv = np.float32(orc.inv127_rz(float(amax)))
            y = (G[t, 128 * j:128 * (j + 1)] * inv).astype(np.float32)
            f = np.floor(y)
            frac = (y - f).astype(np.float32)
            up = Q[t, 128 * j:128 * (j + 1)] == f + 1
            assert np.array_equal(up, u < frac)


def test_bcast_one_direction_per_example(orc):
    """Phi_bcast: every element of an example, all its tokens and channels,
    rounds up exactly when the example's threshold lies below its residual;
    two examples draw different thresholds."""
    rng = np.random.default_rng(8)
    T, N, S = 512, 256, 256
    G = (rng.standard_normal((T, N)) * 1e-2).astype(np.float32)
    Q, delta, _, st = orc.quantize(G, mode=orc.BCAST, seed=9, tensor_id=5, S=S)
    assert st == 0
    us = [orc.example_threshold(b, 9, 5) for b in range(T // S)]
    assert us[0] != us[1]
    for t in range(T):
        for j in range(N // 128):
            d = delta[t // 128, j]
            amax = np.abs(G[128 * (t // 128):128 * (t // 128 + 1), 128 * j:128 * (j + 1)]).max()
            inv = np.float32(orc.inv127_rz(float(amax)))
            y = (G[t, 128 * j:128 * (j + 1)] * inv).astype(np.float32)
            f = np.floor(y)
            frac = (y - f).astype(np.float32)
            assert np.array_equal(Q[t, 128 * j:128 * (j + 1)] == f + 1, us[t // S] < frac)
            assert d == np.float32(amax / np.float32(127))


def test_bcast_unbiased_over_seeds(orc):
    """E[Delta q] = g for every element (Monte Carlo over the example seed)."""
    rng = np.random.default_rng(12)
    G = (rng.standard_normal((128, 128)) * 1e-2).astype(np.float32)
    seeds = 2000
    acc = np.zeros_like(G, dtype=np.float64)
    for sd in range(seeds):
        Q, delta, _, _ = orc.quantize(G, mode=orc.BCAST, seed=sd, tensor_id=0, S=128)
        acc += Q.astype(np.float64) * float(delta[0, 0])
    d = float(delta[0, 0])
    mean = acc / seeds
    sigma = 0.5 * d / np.sqrt(seeds)
    assert np.all(np.abs(mean - G) <= 5 * sigma + 1e-9)


def test_per_tensor_step_is_max_over_tensor(orc):
    rng = np.random.default_rng(2)
    G = (rng.standard_normal((300, 200)) * 1e-2).astype(np.float32)
    G[123, 45] = 0.75
    Q, delta, _, _ = orc.quantize(G, mode=orc.S3R7, seed=1, tile=G.shape)
    assert delta.shape == (1, 1) and delta[0, 0] == np.float32(np.float32(0.75) / np.float32(127))
    assert Q[123, 45] == 127


def test_dw_only_correction_is_the_two_way_dw_and_the_plain_dx(orc):
    """Table II's dW-only row: dX carries no correction, dW the full one."""
    rng = np.random.default_rng(4)
    T, K, N, S = 256, 136, 200, 128
    G = (rng.standard_t(3, size=(T, N)) * 1e-3).astype(np.float32)
    X8 = rng.integers(-127, 128, size=(T, K)).astype(np.int8)
    W8 = rng.integers(-127, 128, size=(K, N)).astype(np.int8)
    s_x = (rng.random(T) * 0.03 + 0.02).astype(np.float32)
    s_w = (rng.random(N) * 5e-4 + 1e-4).astype(np.float32)
    d = orc.linear_backward(G, X8, s_x, W8, s_w, S, orc.S3R, orc.EC_DW_ONLY, seed=3)
    two = orc.linear_backward(G, X8, s_x, W8, s_w, S, orc.S3R, orc.EC_TWO_WAY, seed=3)
    plain = orc.linear_backward(G, X8, s_x, W8, s_w, S, orc.S3R, orc.EC_NONE, seed=3)
    assert np.array_equal(d.dX, plain.dX)
    assert np.array_equal(d.dW, two.dW)
    assert not np.array_equal(d.dW, plain.dW)
