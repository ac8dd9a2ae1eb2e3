"""Pins for the oracle's exact int32 block GEMMs and rescale ([S3R] §III-A: S8
GEMM with S32 accumulation, then rescale).  Checked by brute force against
numpy's int64 matmul, a library routine, on ragged shapes."""
import numpy as np
import pytest


@pytest.mark.parametrize("T,N,K", [(5, 300, 7), (1, 128, 1), (17, 129, 33), (3, 1, 2)])
def test_dx_blocks_brute_force(orc, T, N, K):
    rng = np.random.default_rng(T * 1000 + N)
    Q = rng.integers(-127, 128, size=(T, N)).astype(np.int8)
    W8 = rng.integers(-127, 128, size=(K, N)).astype(np.int8)
    rows = np.arange(T)
    I = orc.dx_blocks(Q, W8, rows)
    full = Q.astype(np.int64) @ W8.astype(np.int64).T
    assert np.array_equal(I.astype(np.int64).sum(2), full)
    for kb in range(I.shape[2]):
        blk = Q[:, kb * 128:(kb + 1) * 128].astype(np.int64) @ W8[:, kb * 128:(kb + 1) * 128].astype(np.int64).T
        assert np.array_equal(I[:, :, kb], blk)


@pytest.mark.parametrize("T,K,N", [(300, 5, 7), (128, 1, 1), (129, 33, 17), (1, 2, 3)])
def test_dw_blocks_brute_force(orc, T, K, N):
    rng = np.random.default_rng(T * 7 + N)
    X8 = rng.integers(-127, 128, size=(T, K)).astype(np.int8)
    Q = rng.integers(-127, 128, size=(T, N)).astype(np.int8)
    J = orc.dw_blocks(X8, Q, np.arange(K))
    full = X8.astype(np.int64).T @ Q.astype(np.int64)
    assert np.array_equal(J.astype(np.int64).sum(2), full)
    for tb in range(J.shape[2]):
        blk = X8[tb * 128:(tb + 1) * 128].astype(np.int64).T @ Q[tb * 128:(tb + 1) * 128].astype(np.int64)
        assert np.array_equal(J[:, :, tb], blk)


def test_worst_case_block_fits_fp32_exactly():
    """A 128-long block of int8 products is bounded by 128 * 127^2 < 2^24, so it
    is an exact fp32 integer (the fact the fp16-carried tensor-core GEMM and the
    per-block rescale rely on)."""
    assert 128 * 127 * 127 < 2 ** 24


def test_rescale_equals_dequantize_then_contract(orc):
    """sum_kb delta * int32-block equals contracting the dequantized codes."""
    rng = np.random.default_rng(7)
    T, N, K = 260, 300, 24
    Q = rng.integers(-127, 128, size=(T, N)).astype(np.int8)
    W8 = rng.integers(-127, 128, size=(K, N)).astype(np.int8)
    X8 = rng.integers(-127, 128, size=(T, K)).astype(np.int8)
    delta = (rng.random((3, 3)) + 0.1).astype(np.float32)
    s_x = (rng.random(T) + 0.5).astype(np.float32)
    s_w = (rng.random(N) + 0.5).astype(np.float32)
    dfull = np.repeat(np.repeat(delta.astype(np.float64), 128, 0), 128, 1)[:T, :N]
    Gt = dfull * Q
    dX = orc.dx(Q, delta, W8, s_x, orc.EC_NONE, None, None, None, T, np.arange(T))
    dW = orc.dw(X8, Q, delta, s_w, orc.EC_NONE, None, None, None, None, T, np.arange(K))
    assert np.allclose(dX, (Gt @ W8.T.astype(np.float64)) / s_x[:, None], rtol=1e-12)
    assert np.allclose(dW, (X8.T.astype(np.float64) @ Gt) / s_w[None, :], rtol=1e-12)
