"""Pins for the oracle's S3R-EC error statistics and correction factors.

Source: "Efficient Quantization Training with Stochastic Rounding via
Structured Subspace Randomness", §III-C ("Subtracting the mean removes the
correlation": the -Z, Z, Z example, 16/9 and 8/9) and §III-D ("Two-way
correction": the orthogonal projection of E_b onto {1_S a^T + c 1_D^T}; what
remains sums to zero along every row and column; the corrected gradients stay
unbiased).  The projection's displayed equations were lost from the page; the
oracle rebuilds them from the prose, and these tests pin the rebuild against
an independent route (a generic least-squares projection) and the stated
invariants.
"""
import numpy as np
import pytest


def test_centering_minus_z_z_z(orc):
    """X1 = -Z, X2 = X3 = Z: after subtracting the mean the first error's
    variance is 16/9 Var(Z) and the average variance is 8/9 Var(Z)."""
    rng = np.random.default_rng(0)
    z = rng.standard_normal(20000).astype(np.float32)
    E = np.stack([-z, z, z], 1)
    eps, _, _ = orc.error_stats(E, 1)
    centered = E.astype(np.float64) - eps[:, None]
    vz = z.astype(np.float64).var()
    v = centered.var(0) / vz
    assert abs(v[0] - 16 / 9) < 1e-6 and abs(v[1] - 4 / 9) < 1e-6 and abs(v[2] - 4 / 9) < 1e-6
    assert abs(v.mean() - 8 / 9) < 1e-6


def _projection(orc, E, S):
    eps, colmean, mu = orc.error_stats(E, S)
    T, N = E.shape
    b = np.arange(T) // S
    return colmean[b] + eps[:, None] - mu[b][:, None], (eps, colmean, mu)


def test_projection_matches_least_squares(orc):
    """P(E_b) equals the least-squares projection of E_b onto the span of
    row-constant and column-constant matrices."""
    rng = np.random.default_rng(1)
    S, N, B = 9, 7, 3
    E = rng.standard_normal((B * S, N)).astype(np.float32)
    P, _ = _projection(orc, E, S)
    for bb in range(B):
        Eb = E[bb * S:(bb + 1) * S].astype(np.float64)
        basis = []
        for n in range(N):
            m = np.zeros((S, N)); m[:, n] = 1; basis.append(m.ravel())
        for s in range(S):
            m = np.zeros((S, N)); m[s, :] = 1; basis.append(m.ravel())
        A = np.stack(basis, 1)
        coef, *_ = np.linalg.lstsq(A, Eb.ravel(), rcond=None)
        Pls = (A @ coef).reshape(S, N)
        assert np.allclose(P[bb * S:(bb + 1) * S], Pls, atol=1e-12)


def test_projection_invariants(orc):
    """Residual sums to zero along every row and every column of each example;
    P is idempotent and the residual is orthogonal to P(E)."""
    rng = np.random.default_rng(2)
    S, N, B = 128, 96, 2
    E = (rng.random((B * S, N)) - 0.5).astype(np.float32)
    P, _ = _projection(orc, E, S)
    R = E.astype(np.float64) - P
    assert np.abs(R.sum(1)).max() < 1e-12
    for bb in range(B):
        assert np.abs(R[bb * S:(bb + 1) * S].sum(0)).max() < 1e-12
    P2, _ = _projection(orc, P.astype(np.float32), S)
    assert np.allclose(P2, P, atol=1e-6)
    assert abs((R * P).sum()) < 1e-9 * np.abs(E).sum()


def _tiny_layer(rng, T, K, N):
    X = rng.standard_normal((T, K)).astype(np.float32)
    W = (rng.standard_normal((K, N)) * 0.02).astype(np.float32)
    G = (rng.standard_t(3, size=(T, N)) * 1e-3).astype(np.float32)
    return X, W, G


@pytest.mark.parametrize("ec_mode", ["EC_NONE", "EC_DX_ONLY", "EC_TWO_WAY", "EC_DX_TOKEN_ONLY"])
def test_factored_correction_equals_dense(orc, ec_mode):
    """The factored corrections (row sums, v_b, xsum_b, p) equal the dense
    (Delta Q - P(E)) W^T / s_x and X^T (Delta Q - P(E)) / s_w, brute force in
    fp64, on a layer with several tiles, two examples and ragged edges."""
    rng = np.random.default_rng(3)
    T, K, N, S, tile = 64, 40, 50, 32, (16, 16)
    X, W, G = _tiny_layer(rng, T, K, N)
    X8, s_x = orc.rtne_operand(X, 0)
    W8, s_w = orc.rtne_operand(W, 1)
    mode = getattr(orc, ec_mode)
    out = orc.linear_backward(G, X8, s_x, W8, s_w, S, mode=orc.S3R, ec_mode=mode, seed=5, tensor_id=1, tile=tile)
    dfull = np.repeat(np.repeat(out.delta.astype(np.float64), tile[0], 0), tile[1], 1)[:T, :N]
    Gt = dfull * out.Q
    P, (eps, _, _) = _projection(orc, out.E, S)
    if mode in (orc.EC_DX_ONLY, orc.EC_TWO_WAY):
        Gx = Gt - P
    elif mode == orc.EC_DX_TOKEN_ONLY:
        Gx = Gt - eps[:, None]
    else:
        Gx = Gt
    Gw = Gt - P if mode == orc.EC_TWO_WAY else Gt
    dX_dense = (Gx @ W8.astype(np.float64).T) / s_x[:, None].astype(np.float64)
    dW_dense = (X8.astype(np.float64).T @ Gw) / s_w[None, :].astype(np.float64)
    assert np.allclose(out.dX, dX_dense, rtol=1e-9, atol=1e-12 * np.abs(dX_dense).max())
    assert np.allclose(out.dW, dW_dense, rtol=1e-9, atol=1e-12 * np.abs(dW_dense).max())


def test_corrected_gradients_unbiased(orc):
    """Mean over seeds of the two-way corrected dX and dW approaches the
    unquantized G' W^T / s_x and X^T G' / s_w ([S3R] §III-D: the correction
    keeps both gradients unbiased)."""
    rng = np.random.default_rng(4)
    T, K, N, S, tile = 32, 12, 24, 16, (16, 8)
    X, W, G = _tiny_layer(rng, T, K, N)
    X8, s_x = orc.rtne_operand(X, 0)
    W8, s_w = orc.rtne_operand(W, 1)
    Gp = (s_x[:, None] * G) * s_w[None, :]
    ref_dx = (Gp.astype(np.float64) @ W8.astype(np.float64).T) / s_x[:, None]
    ref_dw = (X8.astype(np.float64).T @ Gp.astype(np.float64)) / s_w[None, :]
    n = 3000
    acc_x = np.zeros((n, T, K))
    acc_w = np.zeros((n, K, N))
    for s in range(n):
        out = orc.linear_backward(G, X8, s_x, W8, s_w, S, mode=orc.S3R, ec_mode=orc.EC_TWO_WAY, seed=s,
                                  tensor_id=2, tile=tile)
        acc_x[s], acc_w[s] = out.dX, out.dW
    for acc, ref in ((acc_x, ref_dx), (acc_w, ref_dw)):
        se = acc.std(0) / np.sqrt(n)
        ok = se > 0
        z = (acc.mean(0) - ref)[ok] / se[ok]
        assert np.abs(z).max() < 5.5
        assert (np.abs(z) > 3).mean() < 0.02


def test_centered_variance_halves(orc):
    """Evenly spread residuals under a shared threshold: subtracting the token
    mean lowers the average error variance from ~Delta^2/6 to ~Delta^2/12 and
    leaves a non-positive average covariance ([S3R] §III-C)."""
    D = 64
    resid = (np.arange(D) + 0.5) / D
    row = np.concatenate([[127.0], 10.0 + resid]).astype(np.float32)
    G = np.tile(row, (32, 1))
    errs = []
    for seed in range(400):
        _, _, E, _ = orc.quantize(G, mode=orc.S3R, seed=seed)
        e = E[:, 1:].astype(np.float64)
        eps, _, _ = orc.error_stats(E[:, 1:], 1)
        errs.append(e - eps[:, None])
    c = np.cov(np.concatenate(errs, 0), rowvar=False)
    var = np.diag(c).mean()
    off = (c.sum() - np.trace(c)) / (D * (D - 1))
    assert abs(var - 1 / 12) < 0.008, var
    assert off <= 1e-3


def test_ec_factor_integer_parts(orc):
    """rowsum = W8 1 and xsum_b = X8_b^T 1 are exact integers."""
    rng = np.random.default_rng(6)
    W8 = rng.integers(-127, 128, size=(33, 70)).astype(np.int8)
    X8 = rng.integers(-127, 128, size=(40, 33)).astype(np.int8)
    eps = rng.standard_normal(40)
    colmean = rng.standard_normal((2, 70))
    mu = rng.standard_normal(2)
    rowsum, v, xsum, p = orc.ec_factors(eps, colmean, mu, 20, W8, X8)
    assert np.array_equal(rowsum, W8.astype(np.int64).sum(1))
    assert np.array_equal(xsum, X8.astype(np.int64).reshape(2, 20, 33).sum(1))
    assert np.allclose(v, (colmean - mu[:, None]) @ W8.astype(np.float64).T, rtol=1e-12, atol=1e-9)
    assert np.allclose(p, X8.astype(np.float64).T @ eps, rtol=1e-12, atol=1e-9)
