"""Oracle pins for the grouped (mixture-of-experts) mode.

The grouped backward runs the dense SwiGLU block backward per expert over its
slice of the expert-sorted routed rows.  What the grouping itself decides --
tiles and token indices restarting at each group's first row, the tensor ids
16 e + linear, one example per group, empty groups, expert independence -- is
checked here against independently recomputed quantities.
"""
import numpy as np
import pytest

import workloads

E, D, F = 3, 64, 128


def _case(orc, sizes, seed=3):
    rng = np.random.default_rng(seed)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    R = int(offsets[-1])
    f32 = lambda *s, sd=1.0: (rng.standard_normal(s) * sd).astype(np.float32)
    X, a = f32(R, D), f32(R, F)
    W1, W3, W2 = f32(E, D, F, sd=0.02), f32(E, D, F, sd=0.02), f32(E, F, D, sd=0.02)
    h1, h3 = f32(R, F, sd=0.16), f32(R, F, sd=0.16)
    dY = (rng.standard_t(3, size=(R, D)) * 1e-3).astype(np.float32)
    ops = orc.moe_forward_operands(X, W1, W3, W2, a)
    return ops, h1, h3, dY, offsets


def test_single_group_equals_dense(orc):
    """One expert holding every row is the dense block backward (one example,
    tensor ids 0, 1, 2)."""
    ops, h1, h3, dY, _ = _case(orc, [200, 0, 0])
    g = orc.moe_ffn_backward(ops, h1, h3, dY, [0, 200, 200, 200])
    d = orc.ffn_backward(ops.expert(0, 0, 200), h1, h3, dY, 200)
    assert np.array_equal(g.dX, d.dX)
    assert np.array_equal(g.dW1[0], d.dW1) and np.array_equal(g.dW2[0], d.dW2)
    assert not g.dW1[1:].any() and not g.dW2[1:].any() and not g.dW3[1:].any()


def test_tiles_and_thresholds_restart_at_group_offset(orc):
    """Expert 1 starts at row 150 (not a tile boundary): its W2 codes are the
    quantization of its own slice, and every token of the slice rounds in one
    direction relative to u_t recomputed from the Philox definition with the
    token index counted from the group's first row and tensor id 16 + 0."""
    sizes = [150, 170, 60]
    ops, h1, h3, dY, off = _case(orc, sizes)
    g = orc.moe_ffn_backward(ops, h1, h3, dY, off)
    r0, r1 = int(off[1]), int(off[2])
    w2 = g.experts[1].w2
    Q, delta, _, _ = orc.quantize(dY[r0:r1], ops.s_a[r0:r1], ops.s_w2[1], seed=0,
                                  tensor_id=orc.MOE_TID_STRIDE + orc.TID_W2)
    assert np.array_equal(w2.Q, Q) and np.array_equal(w2.delta, delta)
    # every element rounds up iff u_t < p, with u_t recomputed from the Philox
    # definition (token index counted from the group's first row, tensor id
    # 16 + 0) and y = G' * (127 / amax rounded toward zero) in fp32
    Gp = (ops.s_a[r0:r1, None].astype(np.float32) * dY[r0:r1]).astype(np.float32) * ops.s_w2[1][None, :]
    Gp = Gp.astype(np.float32)
    ntr = -(-(r1 - r0) // orc.TILE)
    for i in range(ntr):
        blk = Gp[i * orc.TILE:(i + 1) * orc.TILE]
        inv = np.float32(orc.inv127_rz(float(np.abs(blk).max())))
        y = (blk * inv).astype(np.float32)
        f = np.floor(y)
        p = (y - f).astype(np.float32)
        for j in range(blk.shape[0]):
            u = np.float32(orc.token_threshold(i * orc.TILE + j, 0, orc.MOE_TID_STRIDE + orc.TID_W2))
            up = Q[i * orc.TILE + j] == f[j] + 1
            assert np.array_equal(up, u < p[j])
            assert np.all(up | (Q[i * orc.TILE + j] == f[j]))
    assert ntr == 2
    # the group-local tile grid differs from the global one for this slice
    Qg, dg, _, _ = orc.quantize(dY[:r1], ops.s_a[:r1], ops.s_w2[1], seed=0,
                                tensor_id=orc.MOE_TID_STRIDE + orc.TID_W2)
    assert not np.array_equal(dg[1:], delta[:dg.shape[0] - 1]) or not np.array_equal(Qg[r0:r1], Q)


def test_empty_group_and_expert_independence(orc):
    sizes = [130, 0, 90]
    ops, h1, h3, dY, off = _case(orc, sizes)
    g = orc.moe_ffn_backward(ops, h1, h3, dY, off)
    assert g.experts[1] is None
    assert not g.dW1[1].any() and not g.dW2[1].any() and not g.dW3[1].any()
    # change expert 2's rows only: expert 0's gradients are untouched
    dY2 = dY.copy()
    dY2[off[2]:] *= 3.0
    g2 = orc.moe_ffn_backward(ops, h1, h3, dY2, off)
    assert np.array_equal(g.dX[:off[1]], g2.dX[:off[1]])
    assert np.array_equal(g.dW1[0], g2.dW1[0]) and np.array_equal(g.dW2[0], g2.dW2[0])
    assert not np.array_equal(g.dW2[2], g2.dW2[2])


def test_tensor_ids_differ_per_expert(orc):
    """Two experts with identical rows and weights draw different thresholds
    (tensor ids 0 and 16), so their codes differ somewhere."""
    rng = np.random.default_rng(9)
    rows = 128
    dY = (rng.standard_t(3, size=(rows, D)) * 1e-3).astype(np.float32)
    Q0, _, _, _ = orc.quantize(dY, tensor_id=0)
    Q1, _, _, _ = orc.quantize(dY, tensor_id=orc.MOE_TID_STRIDE)
    assert not np.array_equal(Q0, Q1)


def test_group_sizes_zipf():
    """The routing loads of the MoE workload: Zipf(1.1) over 8 experts,
    largest-remainder rounding (about 39.8% to expert 0, 4.0% to expert 7)."""
    sizes = workloads.moe_group_sizes(32768, 8)
    assert sum(sizes) == 32768
    assert sizes == sorted(sizes, reverse=True)
    assert abs(sizes[0] / 32768 - 0.398) < 0.002 and abs(sizes[7] / 32768 - 0.040) < 0.002
