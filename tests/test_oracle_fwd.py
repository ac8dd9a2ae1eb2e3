"""Pins for the oracle's INT8 forward of the SwiGLU block.

Source: "Efficient Quantization Training with Stochastic Rounding via
Structured Subspace Randomness" -- §III-A (forward operands rounded to
nearest with per-token and per-output-channel scales, Y = diag(s_x) X_hat
W_hat diag(s_w) from S32 (exact integer) accumulation), §IV-A (GEMM outputs rounded to bf16;
the SwiGLU FFN block).
"""
import numpy as np
import pytest
import torch


@pytest.mark.parametrize("T,K,N", [(37, 128, 53), (16, 1000, 24), (5, 4096, 7), (64, 300, 64)])
def test_gemm_fwd_is_the_exact_integer_product_rescaled(orc, T, K, N):
    """Against numpy: the int64 matrix product, converted to float32 (round to
    nearest), then times s_x and s_w in float32."""
    rng = np.random.default_rng(T + K)
    X8 = rng.integers(-127, 128, size=(T, K)).astype(np.int8)
    W8 = rng.integers(-127, 128, size=(K, N)).astype(np.int8)
    s_x = (rng.random(T) * 0.1 + 0.01).astype(np.float32)
    s_w = (rng.random(N) * 0.01 + 0.001).astype(np.float32)
    I = X8.astype(np.int64) @ W8.astype(np.int64)
    exp = ((I.astype(np.float32) * s_x[:, None]).astype(np.float32) * s_w[None, :]).astype(np.float32)
    assert np.array_equal(orc.gemm_fwd(X8, s_x, W8, s_w), exp)


def test_gemm_fwd_saturated_sum_rounds_once(orc):
    """All codes +127 over K = 8192: the sum 8192 * 127^2 = 132,128,768 needs
    27 bits; it is rounded to fp32 once (a blockwise fp32 sum would round on
    the way)."""
    K = 8192
    X8 = np.full((1, K), 127, np.int8)
    W8 = np.full((K, 1), 127, np.int8)
    one = np.ones(1, np.float32)
    y = orc.gemm_fwd(X8, one, W8, one)[0, 0]
    assert y == np.float32(K * 127 * 127)


@pytest.mark.parametrize("T,K,N", [(16, 1000, 24), (5, 4096, 7), (64, 300, 64)])
def test_gemm_fwd_equals_exact_product_within_fp32_bound(orc, T, K, N):
    """Brute force: the exact int64 product scaled in fp64, within three fp32
    roundings (the conversion and the two rescales)."""
    rng = np.random.default_rng(T + K)
    X8 = rng.integers(-127, 128, size=(T, K)).astype(np.int8)
    W8 = rng.integers(-127, 128, size=(K, N)).astype(np.int8)
    s_x = (rng.random(T) + 0.5).astype(np.float32)
    s_w = (rng.random(N) + 0.5).astype(np.float32)
    I = X8.astype(np.int64) @ W8.astype(np.int64)
    exact = I.astype(np.float64) * s_x[:, None].astype(np.float64) * s_w[None, :].astype(np.float64)
    bound = 3 * 2.0 ** -24 * np.abs(exact) + 1e-30
    assert np.all(np.abs(orc.gemm_fwd(X8, s_x, W8, s_w) - exact) <= bound)


def test_float_to_bf16_is_round_to_nearest_even(orc):
    """Equals torch's fp32 -> bf16 conversion (round to nearest even), ties included."""
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(4000) * 10.0 ** rng.integers(-8, 8, 4000)).astype(np.float32)
    ties = np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x3F80FFFF], dtype=np.uint32).view(np.float32)
    x = np.concatenate([x, ties, np.array([0.0, -0.0, np.inf, -np.inf], dtype=np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.to_bf16_bits(x), ref)


def test_swiglu_fwd_matches_torch_reference(orc):
    """h1, h3 rounded to bf16 exactly; a = silu(h1) h3 within one bf16 step of
    torch's fp32 silu (the exp here is the oracle's own, within 2 ulp of libm)."""
    rng = np.random.default_rng(5)
    h1f = (rng.standard_normal(20000) * 2).astype(np.float32)
    h3f = (rng.standard_normal(20000) * 2).astype(np.float32)
    h1b, h3b, ab = orc.swiglu_fwd(h1f, h3f)
    t1 = torch.from_numpy(h1f).to(torch.bfloat16)
    t3 = torch.from_numpy(h3f).to(torch.bfloat16)
    assert np.array_equal(h1b, t1.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(h3b, t3.view(torch.int16).numpy().view(np.uint16))
    ref = (torch.nn.functional.silu(t1.float()) * t3.float())
    a = orc.bf16_to_f32(ab)
    r = ref.numpy()
    ulp = np.abs(r) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(a - r) <= ulp)
    assert np.mean(a == ref.to(torch.bfloat16).float().numpy()) > 0.99


def test_ffn_forward_int8_within_quantization_noise(orc):
    """Y of the INT8 block against the fp64 block on the same bf16 inputs:
    within the RTNE noise of int8 operands; swapping the gate and up weights
    moves it far outside."""
    rng = np.random.default_rng(9)
    T, d, F = 64, 256, 384
    b = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)
    X, W1, W3, W2 = (b(rng.standard_normal((T, d))), b(rng.standard_normal((d, F)) * 0.02),
                     b(rng.standard_normal((d, F)) * 0.02), b(rng.standard_normal((F, d)) * 0.02))
    f = orc.from_torch_bf16
    out = orc.ffn_forward_int8(f(X), f(W1), f(W3), f(W2))
    x, w1, w3, w2 = (t.double().numpy() for t in (X, W1, W3, W2))
    h1, h3 = x @ w1, x @ w3
    ref = (h1 / (1 + np.exp(-h1)) * h3) @ w2
    rel = np.linalg.norm(out.Y - ref) / np.linalg.norm(ref)
    assert rel < 0.03
    sw = orc.ffn_forward_int8(f(X), f(W3), f(W1), f(W2))
    assert np.linalg.norm(sw.Y - ref) / np.linalg.norm(ref) > 0.3
    # the saved activations are the bf16 roundings of the INT8 products
    assert np.array_equal(out.h1, orc.to_bf16_bits(orc.gemm_fwd(out.X8, out.s_x, out.W1_8, out.s_w1)))
