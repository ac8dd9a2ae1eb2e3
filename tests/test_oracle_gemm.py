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


@pytest.mark.parametrize("T,N,K,S", [(260, 300, 24, 130), (128, 128, 1, 128), (1, 129, 3, 1), (300, 257, 40, 150)])
@pytest.mark.parametrize("ec_name", ["EC_NONE", "EC_DX_ONLY", "EC_TWO_WAY", "EC_DX_TOKEN_ONLY", "EC_DW_ONLY"])
def test_matmul_products_equal_loop_products(orc, T, N, K, S, ec_name):
    """dx_matmul / dw_matmul (integer block sums by a library matmul) equal the
    nested-loop dx / dw bit for bit, corrections and rescales included, on
    ragged shapes; rows and krows subsets too."""
    rng = np.random.default_rng(T + 3 * N + 7 * K)
    ec = getattr(orc, ec_name)
    Q = rng.integers(-127, 128, size=(T, N)).astype(np.int8)
    Q[0, :min(N, 5)] = 127                      # extremes of the block sums
    W8 = rng.integers(-127, 128, size=(K, N)).astype(np.int8)
    W8[0, :min(N, 5)] = -127
    X8 = rng.integers(-127, 128, size=(T, K)).astype(np.int8)
    delta = (rng.random((-(-T // 128), -(-N // 128))) + 0.1).astype(np.float32) * np.float32(1e-3)
    s_x = (rng.random(T) + 0.5).astype(np.float32)
    s_w = (rng.random(N) + 0.5).astype(np.float32)
    B = T // S
    eps = rng.standard_normal(T) * 1e-4
    colmean = rng.standard_normal((B, N)) * 1e-4
    mu = rng.standard_normal(B) * 1e-5
    rowsum, v, xsum, p = orc.ec_factors(eps, colmean, mu, S, W8, X8)
    rows = np.arange(T)
    krows = np.arange(K)
    a = orc.dx(Q, delta, W8, s_x, ec, eps, rowsum, v, S, rows)
    b = orc.dx_matmul(Q, delta, W8, s_x, ec, eps, rowsum, v, S, rows, chunk=97)
    assert np.array_equal(a.view(np.uint64), b.view(np.uint64))
    a = orc.dw(X8, Q, delta, s_w, ec, colmean, mu, xsum, p, S, krows)
    b = orc.dw_matmul(X8, Q, delta, s_w, ec, colmean, mu, xsum, p, S, krows)
    assert np.array_equal(a.view(np.uint64), b.view(np.uint64))
    sub = np.array([T - 1, 0]) if T > 1 else np.array([0])
    assert np.array_equal(orc.dx(Q, delta, W8, None, ec, eps, rowsum, v, S, sub),
                          orc.dx_matmul(Q, delta, W8, None, ec, eps, rowsum, v, S, sub))
    ksub = np.array([K - 1, 0]) if K > 1 else np.array([0])
    assert np.array_equal(orc.dw(X8, Q, delta, None, ec, colmean, mu, xsum, p, S, ksub),
                          orc.dw_matmul(X8, Q, delta, None, ec, colmean, mu, xsum, p, S, ksub))


def test_block_sums_exact_at_the_extremes(orc):
    """A 128-long block of +-127 * +-127 products (the largest block sum) is
    exact through the library matmul; a wrong sum trips the guard."""
    A = np.full((3, 128), 127, dtype=np.int8)
    A[1] = -127
    B = np.full((128, 4), 127, dtype=np.int8)
    B[:, 2] = -127
    out = orc.block_sums(A, B)
    assert np.array_equal(out, (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float64))
    assert out[0, 0] == 128 * 127 * 127


def test_ffn_backward_matmul_equals_loops(orc):
    """The FFN block composed with the matmul products equals the loop version
    bit for bit (every intermediate and output)."""
    import workloads
    inp = workloads.ffn_inputs(256, 128, 384, 128, seed=21)
    f = orc.from_torch_bf16
    ops = orc.ffn_forward_operands(f(inp.X), f(inp.W1), f(inp.W3), f(inp.W2), f(inp.a))
    h1, h3, dY = f(inp.h1), f(inp.h3), f(inp.dY)
    a = orc.ffn_backward(ops, h1, h3, dY, 128, orc.S3R, orc.EC_TWO_WAY, seed=3)
    b = orc.ffn_backward(ops, h1, h3, dY, 128, orc.S3R, orc.EC_TWO_WAY, seed=3, matmul=True)
    for k in ("dA", "dX", "dW1", "dW2", "dW3"):
        assert np.array_equal(getattr(a, k), getattr(b, k)), k
    assert np.array_equal(a.w1.Q, b.w1.Q) and np.array_equal(a.w3.Q, b.w3.Q)
