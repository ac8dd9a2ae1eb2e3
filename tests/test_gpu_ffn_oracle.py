"""GPU parity of ffn_backward itself -- the launches the benchmark times --
against the oracle, element by element.

One library call runs the whole block backward: with fp16-carried codes its
products are two mixed tcgen05 launches (dA + dW2, then dX1 + dX3 + dW1 +
dW3), in which every persistent CTA works through many dX and dW tiles in
turn.  The oracle composes the same block from its own pieces; its products
take their integer block sums from a library matmul (equal bit for bit to its
nested loops, see tests/test_oracle_gemm.py), which makes full-size blocks
affordable.

Checked, per block:
  * the codes of dY (Q2) and their tile scales, bit for bit, everywhere;
  * dA (read back from the workspace) and dW2, within the fp32 bound;
  * the codes of dh1 and dh3 (Q1, Q3): equal but for one-step flips where the
    oracle's own decision was a near tie (dA reaches the glue through a
    differently ordered fp32 sum); the exact effect of every flip, and of any
    tile step that moved by an ulp, is added to the oracle's dX, dW1 and dW3
    before they are compared within the fp32 bound.
Sizes: the d=2048 / F=5632 / T=8192 block in full; a ragged mid-size block in
full; the d=4096 / F=14336 / T=16384 block on sampled rows; the MoE workload
on sampled rows of every expert.
"""
import numpy as np
import pytest
import torch

import workloads
from parity_util import (assert_close_mag, codes, dw_magnitude, dx_magnitude, expand_tiles, flip_effect,
                         near_tie_flips, tile_amax)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def s3r():
    import stochastic_rounding_int8_gb300 as m
    m.lib()
    return m


def _host(t):
    return t.detach().cpu().numpy()


def check_block(orc, views, g, ops_o, h1, h3, dY, S, seed, tid_base, rows, krows_d, krows_f, check_dA=True):
    """One block's (or expert's) ffn_backward results against the oracle.
    views: the block's workspace views (codes, tile scales, dA); g: its output
    gradients as host arrays (dX [T, d], dW1 / dW3 [d, F], dW2 [F, d]); rows:
    token rows of dA and dX to compare; krows_d / krows_f: rows of dW1, dW3
    and of dW2; check_dA: False when the glue ran in the dA epilogue (dA is
    not kept)."""
    T = dY.shape[0]
    F = ops_o.A8.shape[1]
    # stage 1: W2
    w2 = orc.linear_backward(dY, ops_o.A8, ops_o.s_a, ops_o.W2_8, ops_o.s_w2, S, orc.S3R, orc.EC_TWO_WAY, seed,
                             tid_base + orc.TID_W2, rows=np.arange(T), krows=krows_f, matmul=True)
    assert w2.status == 0
    assert np.array_equal(codes(views["Q2"]), w2.Q), "codes of dY"
    assert np.array_equal(_host(views["scale2"]), w2.delta), "tile scales of dY"
    if check_dA:
        mdx = dx_magnitude(w2.Q, w2.delta, ops_o.W2_8, ops_o.s_a, w2.eps, w2.rowsum, w2.v, S, rows=rows)
        assert_close_mag(_host(views["dA"])[rows], w2.dX[rows], mdx, "dA")
    mdw = dw_magnitude(ops_o.A8, w2.Q, w2.delta, ops_o.s_w2, w2.colmean, w2.mu, w2.xsum, w2.p, krows=krows_f)
    assert_close_mag(g["dW2"][krows_f], w2.dW, mdw, "dW2")
    # stage 2: the glue on the oracle's own dA, then W1 and W3
    dA = w2.dX.astype(np.float32)
    del w2
    dh1, dh3 = orc.swiglu_bwd(dA, h1, h3)
    del dA
    exp_dx = 0.0
    mag_dx = 0.0
    for name, dh, W8, s_w, tid, qv, sv in (("dW1", dh1, ops_o.W1_8, ops_o.s_w1, orc.TID_W1, "Q1", "scale1"),
                                           ("dW3", dh3, ops_o.W3_8, ops_o.s_w3, orc.TID_W3, "Q3", "scale3")):
        lb = orc.linear_backward(dh, ops_o.X8, ops_o.s_x, W8, s_w, S, orc.S3R, orc.EC_TWO_WAY, seed, tid_base + tid,
                                 rows=rows, krows=krows_d, matmul=True)
        assert lb.status == 0
        Qg, dg = codes(views[qv]), _host(views[sv])
        # the oracle's normalized values y, to judge which decisions were near ties
        gf = (ops_o.s_x[:, None] * dh) * s_w[None, :]
        inv = np.array([orc.inv127_rz(float(a)) for a in tile_amax(gf).ravel()], dtype=np.float32)
        inv = inv.reshape(-(-T // 128), -(-F // 128))
        y = gf * expand_tiles(inv, T, F).astype(np.float32)
        del gf
        u = np.array([orc.token_threshold(t, seed, tid_base + tid) for t in range(T)])[:, None]
        near_tie_flips(Qg, lb.Q, y, u)
        del y
        ddx, ddw = flip_effect(Qg, dg, lb.Q, lb.delta, W8, ops_o.X8, ops_o.s_x, s_w, S, True, True, rows, krows_d)
        exp_dx = exp_dx + lb.dX + ddx
        mag_dx = mag_dx + dx_magnitude(lb.Q, lb.delta, W8, ops_o.s_x, lb.eps, lb.rowsum, lb.v, S, rows=rows)
        mdw = dw_magnitude(ops_o.X8, lb.Q, lb.delta, s_w, lb.colmean, lb.mu, lb.xsum, lb.p, krows=krows_d)
        assert_close_mag(g[name][krows_d], lb.dW + ddw, mdw, name)
        del lb
    assert_close_mag(g["dX"][rows], exp_dx, mag_dx, "dX")


def _run_dense(s3r, orc, T, d, F, S, seed_data, seed, rows=None, krows_d=None, krows_f=None, fuse_glue=False):
    inp = workloads.ffn_inputs(T, d, F, S, seed=seed_data)
    c = lambda t: t.cuda()
    ops = s3r.ffn_forward_operands(c(inp.X), c(inp.W1), c(inp.W3), c(inp.W2), c(inp.a), c(inp.h1), c(inp.h3))
    ws = torch.empty(s3r.ffn_workspace_size(T, d, F, S), dtype=torch.uint8, device="cuda")
    st = s3r.new_status()
    grads = s3r.ffn_backward(ops, c(inp.dY), S, s3r.ROUND_S3R, s3r.EC_TWO_WAY, seed=seed, workspace=ws, status=st,
                             fuse_glue=fuse_glue)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    views = s3r.ffn_workspace_views(ws, T, d, F, S)
    g = {k: _host(getattr(grads, k)) for k in ("dX", "dW1", "dW3", "dW2")}
    for k, v in g.items():
        assert np.isfinite(v).all(), k
    f = orc.from_torch_bf16
    ops_o = orc.ffn_forward_operands(f(inp.X), f(inp.W1), f(inp.W3), f(inp.W2), f(inp.a))
    for name in ("X8", "A8", "W1_8", "W3_8", "W2_8"):
        assert np.array_equal(codes(getattr(ops, name)), getattr(ops_o, name)), name
    for name in ("s_x", "s_a", "s_w1", "s_w3", "s_w2"):
        assert np.array_equal(_host(getattr(ops, name)), getattr(ops_o, name)), name
    del ops
    rows = np.arange(T) if rows is None else rows
    krows_d = np.arange(d) if krows_d is None else krows_d
    krows_f = np.arange(F) if krows_f is None else krows_f
    check_block(orc, views, g, ops_o, f(inp.h1), f(inp.h3), f(inp.dY), S, seed, 0, rows, krows_d, krows_f,
                check_dA=not fuse_glue)


def test_ffn_backward_block_in_full(s3r, orc):
    """d=2048, F=5632, T=8192 (4 x 2048 tokens), S3R-EC two-way, exactly as the
    benchmark's context runs it: every element of dA, dX, dW1, dW3 and dW2.
    The dA + dW2 launch gives each of the persistent CTAs about 12 tiles, the
    dX1 + dX3 + dW1 + dW3 launch about 6, dX and dW tiles mixed."""
    _run_dense(s3r, orc, 8192, 2048, 5632, 2048, workloads.DATA_SEED + 1, seed=0)


def test_ffn_backward_ragged_block_in_full(s3r, orc):
    """A mid-size block with ragged tiles on every GEMM edge (T = 3 x 640,
    d = 520, F = 1416: neither width a multiple of 128 or 256)."""
    _run_dense(s3r, orc, 1920, 520, 1416, 640, 77, seed=3)


def test_ffn_backward_fused_glue_block_in_full(s3r, orc):
    """The same d=2048 block with the SwiGLU glue and the quantization of dh1,
    dh3 inside the dA GEMM's epilogue (fuse_glue): every code of Q1, Q3
    judged against the oracle's glue on its own dA, and every element of dX,
    dW1, dW3, dW2."""
    _run_dense(s3r, orc, 8192, 2048, 5632, 2048, workloads.DATA_SEED + 1, seed=0, fuse_glue=True)


def test_ffn_backward_fused_glue_ragged_block_in_full(s3r, orc):
    """The ragged mid-size block with the fused glue (the last 256-wide dA tile
    keeps 8 valid columns in its second half: F = 1416)."""
    _run_dense(s3r, orc, 1920, 520, 1416, 640, 77, seed=3, fuse_glue=True)


def test_ffn_backward_large_block_sampled(s3r, orc):
    """d=4096, F=14336, T=16384 (8 x 2048 tokens), S3R-EC two-way, the
    benchmark's timed block: all codes, and dA, dX, dW1, dW3, dW2 on sampled
    rows (each row compared in full), first and last rows included."""
    T, d, F = 16384, 4096, 14336
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([[0, 127, 128, 2047, 2048, T - 1], rng.choice(T, 26, replace=False)]))
    krows_d = np.unique(np.concatenate([[0, d - 1], rng.choice(d, 14, replace=False)]))
    krows_f = np.unique(np.concatenate([[0, F - 1], rng.choice(F, 14, replace=False)]))
    _run_dense(s3r, orc, T, d, F, 2048, workloads.DATA_SEED + 2, seed=1, rows=rows, krows_d=krows_d,
               krows_f=krows_f)


def test_moe_backward_every_expert_sampled(s3r, orc):
    """The MoE workload at full size (8 experts, d=4096, F=1408, 16384 tokens
    top-2, Zipf(1.1) loads: 32768 routed rows), grouped S3R-EC two-way through
    one ffn_backward call: for every expert, all of its codes and dA, a whole
    128-row block of its dX rows plus sampled rows, and sampled rows of its
    dW1, dW3 (including a whole 128-row block) and dW2."""
    w = workloads.WORKLOADS["moe_e8_d4096_F1408_tok16384_top2"]
    d, F = w["d"], w["F"]
    inp = workloads.moe_inputs(w["tokens"], w["topk"], w["experts"], d, F, seed=workloads.DATA_SEED + 5)
    offs = inp.offsets
    c = lambda t: t.cuda()
    ops = s3r.moe_forward_operands(c(inp.X), c(inp.W1), c(inp.W3), c(inp.W2), c(inp.a), c(inp.h1), c(inp.h3))
    ws = torch.empty(s3r.grouped_workspace_size(offs, d, F), dtype=torch.uint8, device="cuda")
    st = s3r.new_status()
    grads = s3r.ffn_backward(ops, c(inp.dY), 0, s3r.ROUND_S3R, s3r.EC_TWO_WAY, seed=2, workspace=ws, status=st,
                             group_offsets=offs)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    f = orc.from_torch_bf16
    ops_o = orc.moe_forward_operands(f(inp.X), f(inp.W1), f(inp.W3), f(inp.W2), f(inp.a))
    assert np.array_equal(codes(ops.A8), ops_o.A8) and np.array_equal(codes(ops.W2_8), ops_o.W2_8)
    assert np.array_equal(_host(ops.s_w1), ops_o.s_w1) and np.array_equal(_host(ops.s_a), ops_o.s_a)
    del ops
    h1, h3, dY = f(inp.h1), f(inp.h3), f(inp.dY)
    gh = {k: getattr(grads, k) for k in ("dX", "dW1", "dW3", "dW2")}
    rng = np.random.default_rng(5)
    for e in range(w["experts"]):
        r0, r1 = offs[e], offs[e + 1]
        Tg = r1 - r0
        assert Tg > 0
        views = s3r.ffn_workspace_views(ws, Tg, d, F, Tg, group_offsets=offs, group=e)
        g = {"dX": _host(gh["dX"][r0:r1]), "dW1": _host(gh["dW1"][e]), "dW3": _host(gh["dW3"][e]),
             "dW2": _host(gh["dW2"][e])}
        blk = (Tg // 2) // 128 * 128
        rows = np.unique(np.concatenate([np.arange(blk, min(Tg, blk + 128)), [0, Tg - 1],
                                         rng.choice(Tg, 6, replace=False)]))
        krows_d = np.unique(np.concatenate([np.arange(128, 256), [0, d - 1], rng.choice(d, 4, replace=False)]))
        krows_f = np.unique(np.concatenate([[0, F - 1], rng.choice(F, 6, replace=False)]))
        check_block(orc, views, g, ops_o.expert(e, r0, r1), h1[r0:r1], h3[r0:r1], dY[r0:r1], Tg, 2,
                    orc.MOE_TID_STRIDE * e, rows, krows_d, krows_f)
