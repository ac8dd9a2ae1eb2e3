"""CPU checks of the GPU tests' comparison helpers: the streamed code-flip
effect equals the dense formula (the difference D through the per-example
projection and both products), and the vectorized tile absmax equals a loop."""
import numpy as np

from parity_util import TILE, expand_tiles, flip_effect, projection, tile_amax


def _dense(Qg, dg, Qo, do, W8, X8, s_x, s_w, S, dx_ec, dw_ec):
    T, N = Qg.shape
    D = expand_tiles(dg, T, N) * Qg - expand_tiles(do, T, N) * Qo
    Dx = D - projection(D, S) if dx_ec else D
    Dw = D - projection(D, S) if dw_ec else D
    return (Dx @ W8.astype(np.float64).T) / s_x[:, None], (X8.astype(np.float64).T @ Dw) / s_w[None, :]


def test_flip_effect_equals_dense_formula():
    rng = np.random.default_rng(4)
    T, N, K, S = 768, 300, 40, 256
    Qo = rng.integers(-127, 128, size=(T, N)).astype(np.int8)
    Qg = Qo.copy()
    flips = rng.random((T, N)) < 0.01
    Qg[flips] = np.clip(Qg[flips].astype(np.int32) + rng.choice([-1, 1], flips.sum()), -127, 127)
    do = (rng.random((-(-T // TILE), -(-N // TILE))) + 0.1).astype(np.float32)
    dg = do.copy()
    dg[1, 2] = np.nextafter(dg[1, 2], np.float32(1))   # one tile whose step differs by an ulp
    W8 = rng.integers(-127, 128, size=(K, N)).astype(np.int8)
    X8 = rng.integers(-127, 128, size=(T, K)).astype(np.int8)
    s_x = (rng.random(T) + 0.5).astype(np.float32)
    s_w = (rng.random(N) + 0.5).astype(np.float32)
    rows = np.array([0, 5, 300, T - 1])
    krows = np.array([K - 1, 3, 0])
    for dx_ec, dw_ec in ((True, True), (True, False), (False, False), (False, True)):
        ddx, ddw = flip_effect(Qg, dg, Qo, do, W8, X8, s_x, s_w, S, dx_ec, dw_ec, rows, krows, chunk=256)
        ex, ew = _dense(Qg, dg, Qo, do, W8, X8, s_x.astype(np.float64), s_w.astype(np.float64), S, dx_ec, dw_ec)
        assert np.allclose(ddx, ex[rows], rtol=1e-10, atol=1e-9 * np.abs(ex).max())
        assert np.allclose(ddw, ew[krows], rtol=1e-10, atol=1e-9 * np.abs(ew).max())


def test_tile_amax_equals_loop():
    rng = np.random.default_rng(5)
    g = rng.standard_normal((300, 257)).astype(np.float32)
    got = tile_amax(g)
    for i in range(got.shape[0]):
        for j in range(got.shape[1]):
            assert got[i, j] == np.abs(g[i * TILE:(i + 1) * TILE, j * TILE:(j + 1) * TILE]).max()
