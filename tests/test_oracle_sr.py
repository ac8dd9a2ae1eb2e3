"""Pins for the oracle's quantizers (S3R, independent SR, RTNE).

Sources: "Stochastic Rounding" (transformer-math blog) -- the definition, the
probability formula, unbiasedness, the variance bound and the 256.3 worked
example; "Efficient Quantization Training with Stochastic Rounding via
Structured Subspace Randomness" -- §III-A (SR operator, RTNE forward operands,
per-tensor step max|G'|/127), §III-B (shared per-token thresholds), §III-C
(same-direction rounding, variance ~ Delta^2/6 and covariance ~ Delta^2/12 for
evenly spread residuals).
"""
import json
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sr_worked_example.json")
SEEDS = 10_000


@pytest.fixture(scope="module")
def ex():
    with open(GOLDEN) as f:
        return json.load(f)


def test_worked_example_single_step(orc, ex):
    x = np.float32(ex["x"])
    p = float(x) - math.floor(float(x))        # frac(256.3f): 0.29998779296875
    assert abs(p - ex["p_page"]) < 1e-4
    assert orc.sr_step(x, 0.0) == ex["x_hi"]
    assert orc.sr_step(x, p - 2 ** -24) == ex["x_hi"]
    assert orc.sr_step(x, p) == ex["x_lo"]       # "u < p" rounds up; u = p does not
    assert orc.sr_step(x, 0.9) == ex["x_lo"]
    # on the grid: p = 0 never moves
    assert orc.sr_step(np.float32(256.0), 0.0) == 256.0


def test_worked_example_rtn_freezes_and_sr_walk(orc, ex):
    """RTN keeps w = 256 forever; the SR walk's mean after 10 steps is 259."""
    w0, g, steps = ex["x_lo"], np.float32(ex["update_per_step"]), ex["steps"]
    # RTN through the oracle's RTNE quantizer with a step of exactly 1
    # (tile amax 127 => Delta = 1, inverse = 1); 256.3 is shifted by -156 into
    # the int8 range with the same fractional part.
    G = np.array([[127.0, np.float32(w0 - 156 + float(g))]], dtype=np.float32)
    Q, delta, _, st = orc.quantize(G, mode=orc.RTNE)
    assert st == 0 and delta[0, 0] == 1.0 and Q[0, 1] == w0 - 156 == 100
    finals = np.empty(SEEDS)
    for trial in range(SEEDS):
        w = np.float32(w0)
        for s in range(steps):
            u = orc.token_threshold(s, trial, 99)
            w = np.float32(orc.sr_step(np.float32(w + g), u))
        finals[trial] = w
    p = float(np.float32(w0) + g) - w0
    sigma = math.sqrt(steps * p * (1 - p) / SEEDS)
    assert abs(finals.mean() - ex["expected_after_steps"]) < 3 * sigma + steps * 2e-5
    assert abs(sigma - 0.0145) < 1e-3


def test_paper_example_point_three(orc, ex):
    """0.3 with step 1 rounds to 1 with probability 0.3 (S3R quantizer path)."""
    pe = ex["paper_example"]
    G = np.array([[127.0, pe["x"]]], dtype=np.float32)
    ups = 0
    for seed in range(SEEDS):
        Q, delta, _, _ = orc.quantize(G, mode=orc.S3R, seed=seed)
        assert delta[0, 0] == pe["step"]
        assert Q[0, 1] in (0, 1)
        ups += int(Q[0, 1] == 1)
    p = float(np.float32(pe["x"]))
    assert abs(ups / SEEDS - pe["probability"]) < 3 * math.sqrt(p * (1 - p) / SEEDS)


def _mc(orc, G, mode, n=SEEDS, **kw):
    codes = np.empty((n,) + G.shape, dtype=np.int8)
    delta = None
    for s in range(n):
        Q, d, _, st = orc.quantize(G, mode=mode, seed=s, **kw)
        assert st == 0
        codes[s] = Q
        delta = d
    return codes, delta


@pytest.mark.parametrize("mode", ["S3R", "INDEP"])
def test_unbiased_and_variance(orc, mode):
    """E[SR(x)] = x and Var = p(1-p) Delta^2 (blog: "Why it is unbiased",
    "The variance cost of the trade"), per element over 10^4 seeds."""
    rng = np.random.default_rng(11)
    G = (rng.standard_normal((8, 24)) * 0.01).astype(np.float32)
    codes, delta = _mc(orc, G, getattr(orc, mode), n=4000)
    d = float(delta[0, 0])
    inv = np.float32(orc.inv127_rz(float(np.abs(G).max())))
    y = (G * inv).astype(np.float64)            # the value SR sees, in grid units
    p = y - np.floor(y)
    mean = codes.astype(np.float64).mean(0)
    var_theory = p * (1 - p)
    se = np.sqrt(np.maximum(var_theory, 1e-30) / codes.shape[0])
    z = (mean - y) / se                         # E[SR(y)] = y
    n = codes.shape[0]
    ok = n * var_theory >= 5                    # where the normal approximation holds
    assert np.abs(z[ok]).max() < 5.0
    assert (np.abs(z[ok]) > 3).mean() < 0.02
    # near-certain elements: the count of the rare outcome stays within a Poisson tail
    rare = (var_theory > 0) & ~ok
    lam = n * np.minimum(p, 1 - p)[rare]
    f = np.floor(y)[rare]
    ups = (codes[:, rare] > f).sum(0)
    minority = np.where(p[rare] < 0.5, ups, n - ups)
    assert (minority <= lam + 6 * np.sqrt(lam) + 4).all()
    var_emp = codes.astype(np.float64).var(0)
    rel = np.abs(var_emp[ok] - var_theory[ok]) / var_theory[ok]
    assert np.median(rel) < 0.05
    assert (var_theory <= 0.25 + 1e-12).all()
    # dequantizing by delta returns G' up to fp32 rounding: |delta * inv - 1| <= 2^-22
    assert abs(np.float64(delta[0, 0]) * np.float64(inv) - 1.0) <= 2.0 ** -22


@pytest.mark.parametrize("mode", ["S3R", "INDEP"])
def test_dequantized_codes_are_unbiased(orc, mode):
    """E[Delta q] = G' (blog: "Why it is unbiased"), directly on the dequantized
    code, within what the fp32 arithmetic allows: the normalizer 127/amax is
    rounded toward zero and Delta = amax/127 to nearest, so Delta * y differs
    from G' by at most 2^-21 |G'| (|Delta * inv - 1| <= 2^-22, plus the
    rounding of y), and the 24-bit threshold grid adds at most 2^-24 Delta.
    Checked two ways: the mean of Delta q over 4000 seeds (5 sigma plus that
    bound), and the exact expectation Delta (floor(y) + P(up)) with P(up) =
    ceil(p 2^24) / 2^24 the law of u < p on the grid, against the bound alone."""
    rng = np.random.default_rng(12)
    G = (rng.standard_normal((8, 24)) * 0.01).astype(np.float32)
    G[3, 5] = np.float32(0.045)                 # the amax element, coded near 127
    codes, delta = _mc(orc, G, getattr(orc, mode), n=4000)
    d = np.float64(delta[0, 0])
    bound = 2.0 ** -21 * np.abs(G.astype(np.float64)) + 2.0 ** -24 * d
    deq = d * codes.astype(np.float64)
    mean = deq.mean(0)
    se = deq.std(0) / np.sqrt(codes.shape[0]) + 1e-30
    assert (np.abs(mean - G) <= 5 * se + bound).all()
    inv = np.float32(orc.inv127_rz(float(np.abs(G).max())))
    y = (G * inv).astype(np.float64)
    f = np.floor(y)
    p_up = np.ceil((y - f) * 2.0 ** 24) / 2.0 ** 24
    expect = d * (f + p_up)
    assert (np.abs(expect - G) <= bound).all()
    assert np.abs(expect - G).max() > 0          # the bound is not vacuous: fp32 leaves a (tiny) bias


def test_on_grid_values_unchanged(orc):
    """Values already on the grid never move ("If x is already on the grid,
    p = 0 and SR leaves it alone")."""
    rng = np.random.default_rng(3)
    for j in (-20, -3, 0, 4):
        k = rng.integers(-127, 128, size=(130, 257)).astype(np.float32)
        k[0, 0] = 127.0
        G = k * np.float32(2.0 ** j)
        for mode in (orc.S3R, orc.INDEP, orc.RTNE):
            for seed in (0, 1, 12345):
                Q, delta, E, st = orc.quantize(G, mode=mode, seed=seed)
                assert st == 0
                # every tile whose amax is 127*2^j has Delta = 2^j exactly
                assert delta[0, 0] == 2.0 ** j
                assert np.array_equal(Q[:128, :128], k[:128, :128].astype(np.int8))
                assert np.all(E[:128, :128] == 0.0)


def test_same_direction_per_token(orc):
    """A shared threshold rounds a token's elements in a common direction: every
    rounded-up element has a larger residual than every rounded-down one
    ([S3R] §III-C "Broadcasting makes the errors move together")."""
    rng = np.random.default_rng(4)
    G = (rng.standard_normal((256, 384)) * 1e-3).astype(np.float32)
    Q, delta, E, _ = orc.quantize(G, mode=orc.S3R, seed=7)
    inv = np.float32(orc.inv127_rz(float(np.abs(G[:128, :128]).max())))
    y = G[:128, :128] * inv
    f = np.floor(y)
    p = y - f
    up = Q[:128, :128].astype(np.float32) == f + 1
    mixed = 0
    for t in range(128):
        if up[t].any() and (~up[t]).any():
            mixed += 1
            assert p[t][up[t]].min() > p[t][~up[t]].max()
    assert mixed > 100
    # independent SR has no such order
    Qi, _, _, _ = orc.quantize(G, mode=orc.INDEP, seed=7)
    upi = Qi[:128, :128].astype(np.float32) == f + 1
    viol = sum(1 for t in range(128) if upi[t].any() and (~upi[t]).any() and p[t][upi[t]].min() < p[t][~upi[t]].max())
    assert viol > 100


def test_shared_threshold_covariance(orc):
    """Evenly spread residuals: Var(e) ~ Delta^2/6 and mean pairwise covariance
    ~ Delta^2/12 under a shared threshold; ~0 under independent thresholds
    ([S3R] §III-C)."""
    D = 64
    resid = (np.arange(D) + 0.5) / D
    row = np.concatenate([[127.0], 10.0 + resid]).astype(np.float32)   # Delta = 1
    G = np.tile(row, (64, 1))                                           # 64 tokens
    for mode, want_cov in (("S3R", 1 / 12), ("INDEP", 0.0)):
        errs = []
        for seed in range(300):
            _, delta, E, _ = orc.quantize(G, mode=getattr(orc, mode), seed=seed)
            assert delta[0, 0] == 1.0
            errs.append(E[:, 1:].astype(np.float64))
        e = np.concatenate(errs, 0)           # samples x D
        cov = np.cov(e, rowvar=False)
        var = np.diag(cov).mean()
        off = (cov.sum() - np.trace(cov)) / (D * (D - 1))
        assert abs(var - 1 / 6) < 0.01, (mode, var)
        assert abs(off - want_cov) < 0.01, (mode, off)


def test_rtne_ties_to_even_and_clamp(orc):
    G = np.array([[127.0, 2.5, 3.5, -2.5, 0.5, -0.5, 126.5, -127.0]], dtype=np.float32)
    Q, delta, _, _ = orc.quantize(G, mode=orc.RTNE)
    assert delta[0, 0] == 1.0
    assert Q.tolist() == [[127, 2, 4, -2, 0, 0, 126, -127]]
    assert np.array_equal(Q.astype(np.float64), np.rint(G.astype(np.float64)))


def test_clamp_never_minus_128(orc):
    rng = np.random.default_rng(8)
    G = (rng.standard_t(3, size=(300, 300)) * 1e-3).astype(np.float32)
    for mode in (orc.S3R, orc.INDEP, orc.RTNE):
        for seed in range(5):
            Q, delta, E, _ = orc.quantize(G, mode=mode, seed=seed)
            assert Q.min() >= -127 and Q.max() <= 127
            # the element carrying the tile amax codes to +-127 (or +-126 if it rounds down)
            ti = np.abs(G[:128, :128]).argmax()
            assert abs(int(Q[:128, :128].flat[ti])) >= 126


def test_per_tensor_step_special_case(orc):
    """tile = whole tensor reproduces the paper's per-tensor step max|G'|/127."""
    rng = np.random.default_rng(9)
    T, N = 200, 300
    G = (rng.standard_normal((T, N)) * 1e-3).astype(np.float32)
    s_x = (rng.random(T) + 0.5).astype(np.float32)
    s_w = (rng.random(N) + 0.5).astype(np.float32)
    Q, delta, _, _ = orc.quantize(G, s_x, s_w, mode=orc.S3R, tile=(T, N))
    Gp = (s_x[:, None] * G) * s_w[None, :]
    assert delta.shape == (1, 1)
    assert delta[0, 0] == np.float32(np.abs(Gp).max()) / np.float32(127.0)


def test_zero_tile_and_nonfinite(orc):
    G = np.zeros((130, 130), dtype=np.float32)
    G[129, 129] = 1.0
    Q, delta, E, st = orc.quantize(G, mode=orc.S3R)
    assert st == 0 and delta[0, 0] == 0.0 and not Q[:128, :128].any() and not E[:128, :128].any()
    assert delta[1, 1] == np.float32(1.0) / np.float32(127.0) and Q[129, 129] == 127
    G[5, 5] = np.nan
    _, delta, _, st = orc.quantize(G, mode=orc.S3R)
    assert st == -4 and np.isnan(delta[0, 0]) and delta[1, 1] > 0


def test_error_definition_and_partials(orc):
    """E = Delta*Q - G' ([S3R] §III-A) and the tile partial sums of E."""
    rng = np.random.default_rng(10)
    T, N = 300, 260
    G = (rng.standard_normal((T, N)) * 1e-2).astype(np.float32)
    Q, delta, E, _ = orc.quantize(G, mode=orc.S3R, seed=3)
    dfull = np.repeat(np.repeat(delta.astype(np.float64), 128, 0), 128, 1)[:T, :N]
    assert np.allclose(E, dfull * Q - G, rtol=0, atol=1e-7 * np.abs(G).max())
    assert np.all(np.abs(E) <= dfull * (1 + 1e-6))
    tok, col = orc.error_partials(E)
    for j in range(tok.shape[1]):
        assert np.allclose(tok[:, j], E[:, j * 128:(j + 1) * 128].astype(np.float64).sum(1), atol=1e-12)
    for i in range(col.shape[0]):
        assert np.allclose(col[i], E[i * 128:(i + 1) * 128].astype(np.float64).sum(0), atol=1e-12)


def test_rtne_operand_scales(orc):
    """Forward operands: X ~ diag(s_x) X_hat, W ~ W_hat diag(s_w) with RTNE
    ([S3R] §III-A)."""
    rng = np.random.default_rng(12)
    A = rng.standard_normal((40, 70)).astype(np.float32)
    A[3] = 0.0
    Q, s = orc.rtne_operand(A, 0)
    assert s[3] == 1.0 and not Q[3].any()
    for r in range(40):
        if r == 3:
            continue
        assert s[r] == np.float32(np.abs(A[r]).max()) / np.float32(127)
        assert np.abs(Q[r]).max() == 127 and Q.min() >= -127
    recon = Q.astype(np.float64) * s[:, None]
    assert np.all(np.abs(recon - A) <= 0.5 * s[:, None] * (1 + 1e-5))
    Qc, sc = orc.rtne_operand(A, 1)
    recon = Qc.astype(np.float64) * sc[None, :]
    assert np.all(np.abs(recon - A) <= 0.5 * sc[None, :] * (1 + 1e-5))
    # ties go to even
    B = np.array([[127.0, 2.5, -3.5, 0.5]], dtype=np.float32)
    Qb, sb = orc.rtne_operand(B, 0)
    assert sb[0] == 1.0 and Qb.tolist() == [[127, 2, -4, 0]]


def test_window_equals_slice_of_full(orc):
    """Quantizing a tile-aligned window with global indices reproduces the
    corresponding slice of the whole tensor's quantization (used by the
    sampled full-size parity tests)."""
    rng = np.random.default_rng(13)
    T, N = 384, 300
    G = (rng.standard_t(3, size=(T, N)) * 1e-3).astype(np.float32)
    for mode in (orc.S3R, orc.INDEP, orc.RTNE):
        Q, delta, E, _ = orc.quantize(G, mode=mode, seed=21, tensor_id=4)
        Qw, dw, Ew, _ = orc.quantize(G[128:256, 128:300], mode=mode, seed=21, tensor_id=4, window=(128, 128, N))
        assert np.array_equal(Qw, Q[128:256, 128:300])
        assert np.array_equal(dw, delta[1:2, 1:3])
        assert np.array_equal(Ew, E[128:256, 128:300])


def test_inverse_rounds_toward_zero_and_bounds_y(orc):
    """inv = 127/amax rounded toward zero: never above the exact quotient, at
    most one ulp below it (checked against exact rational arithmetic), so
    |g * inv| <= 127 for every |g| <= amax and codes never need clamping."""
    from fractions import Fraction
    rng = np.random.default_rng(21)
    amaxes = np.concatenate([rng.random(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, 20000),
                             np.float32([1.0, 127.0, 3.0, 1e-38, 3e38, 0.1])]).astype(np.float32)
    for a in amaxes[:4000]:
        a = np.float32(a)
        if not np.isfinite(a) or a <= 0:
            continue
        inv = np.float32(orc.inv127_rz(float(a)))
        exact = Fraction(127) / Fraction(float(a))
        assert Fraction(float(inv)) <= exact
        assert Fraction(float(np.nextafter(inv, np.float32(np.inf)))) > exact
    for a in amaxes:
        a = np.float32(a)
        if not np.isfinite(a) or a <= 0:
            continue
        inv = np.float32(orc.inv127_rz(float(a)))
        assert abs(np.float32(a) * inv) <= np.float32(127.0)
        assert abs(np.float32(-a) * inv) <= np.float32(127.0)
