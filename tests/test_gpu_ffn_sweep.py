"""GPU: ffn_backward on seeded random shapes, every element against the oracle.

The fixed shapes of test_gpu_ffn_oracle.py are joined here by a seeded sweep
of ragged blocks: widths that are multiples of 8 but rarely of 128 or 256,
token counts that split into one or several examples, and grouped calls with
empty, one-row, 127-, 128- and 129-row experts.  Each case runs the
library's own launches (the mixed tcgen05 GEMMs with their static tile deal,
partial tiles on every edge) and is compared in full with the oracle through
the same checks as the fixed shapes.
"""
import numpy as np
import pytest
import torch

import workloads
from parity_util import codes
from test_gpu_ffn_oracle import _host, _run_dense, check_block

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def s3r():
    import stochastic_rounding_int8_gb300 as m
    m.lib()
    return m


def _shapes(n, seed=2025):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        d = 8 * int(rng.integers(2, 81))        # 16 .. 640
        F = 8 * int(rng.integers(2, 201))       # 16 .. 1600
        B = int(rng.integers(1, 4))
        if rng.random() < 0.3:
            S = int(rng.integers(1, 700))       # one example of any length
            B = 1
        else:
            S = 128 * int(rng.integers(1, 5))
        out.append((B * S, d, F, S, int(rng.integers(0, 1 << 30))))
    return out


@pytest.mark.parametrize("T,d,F,S,seed", _shapes(16))
def test_random_dense_block_in_full(s3r, orc, T, d, F, S, seed):
    _run_dense(s3r, orc, T, d, F, S, seed % 1000, seed=seed % 97)


@pytest.mark.parametrize("d,F,sizes,data_seed", [
    (136, 392, [129, 0, 1, 128, 127, 300, 0, 64], 71),
    (264, 1416, [513, 2, 255, 256, 0, 17], 72),
])
def test_random_grouped_block_every_expert_in_full(s3r, orc, d, F, sizes, data_seed):
    inp = workloads.moe_inputs_sized(sizes, d, F, seed=data_seed)
    offs = inp.offsets
    c = lambda t: t.cuda()
    ops = s3r.moe_forward_operands(c(inp.X), c(inp.W1), c(inp.W3), c(inp.W2), c(inp.a), c(inp.h1), c(inp.h3))
    ws = torch.empty(s3r.grouped_workspace_size(offs, d, F), dtype=torch.uint8, device="cuda")
    st = s3r.new_status()
    grads = s3r.ffn_backward(ops, c(inp.dY), 0, s3r.ROUND_S3R, s3r.EC_TWO_WAY, seed=6, workspace=ws, status=st,
                             group_offsets=offs)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    f = orc.from_torch_bf16
    ops_o = orc.moe_forward_operands(f(inp.X), f(inp.W1), f(inp.W3), f(inp.W2), f(inp.a))
    assert np.array_equal(codes(ops.A8), ops_o.A8) and np.array_equal(codes(ops.X8), ops_o.X8)
    del ops
    h1, h3, dY = f(inp.h1), f(inp.h3), f(inp.dY)
    for e in range(len(sizes)):
        r0, r1 = offs[e], offs[e + 1]
        Tg = r1 - r0
        g = {"dX": _host(grads.dX[r0:r1]), "dW1": _host(grads.dW1[e]), "dW3": _host(grads.dW3[e]),
             "dW2": _host(grads.dW2[e])}
        if Tg == 0:   # an expert without rows has zero weight gradients
            assert not g["dW1"].any() and not g["dW3"].any() and not g["dW2"].any()
            continue
        views = s3r.ffn_workspace_views(ws, Tg, d, F, Tg, group_offsets=offs, group=e)
        check_block(orc, views, g, ops_o.expert(e, r0, r1), h1[r0:r1], h3[r0:r1], dY[r0:r1], Tg, 6,
                    orc.MOE_TID_STRIDE * e, np.arange(Tg), np.arange(d), np.arange(F))
