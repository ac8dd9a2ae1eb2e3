"""GPU: ffn_backward captured in a CUDA graph.

A training loop replays its step as a CUDA graph to drop the host's launch
work.  ffn_backward launches every kernel on the caller's stream (grouped mode
forks per-expert steps onto side streams and joins them back with events,
which a capture records as graph edges), allocates nothing and never
synchronizes, so after one eager call (which sets the kernels' attributes and
creates the side streams) it can be captured.  Each replay, over new upstream
gradients written into the captured input, must equal an eager call on the
same inputs bit for bit.
"""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def s3r():
    import stochastic_rounding_int8_gb300 as m
    m.lib()
    return m


def _check_capture(s3r, ops, dY, S, group_offsets, n_new=2, seed=9):
    T, d = dY.shape
    F = ops.A8.shape[1]
    if group_offsets is None:
        grads = s3r.alloc_ffn_grads(T, d, F)
        ws = torch.empty(s3r.ffn_workspace_size(T, d, F, S), dtype=torch.uint8, device="cuda")
    else:
        grads = s3r.alloc_moe_grads(T, len(group_offsets) - 1, d, F, "cuda")
        ws = torch.empty(s3r.grouped_workspace_size(group_offsets, d, F), dtype=torch.uint8, device="cuda")
    st = s3r.new_status()
    x = dY.clone()   # the captured input
    call = lambda g, w: s3r.ffn_backward(ops, x, S, seed=seed, grads=g, workspace=w, status=st,
                                         group_offsets=group_offsets)
    call(grads, ws)   # eager warm-up
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call(grads, ws)
    ref_grads = (s3r.alloc_ffn_grads(T, d, F) if group_offsets is None
                 else s3r.alloc_moe_grads(T, len(group_offsets) - 1, d, F, "cuda"))
    ref_ws = torch.empty_like(ws)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1234)
    for i in range(n_new):
        if i:
            x.copy_((torch.randn(x.shape, generator=gen, device="cuda") * 1e-3).to(torch.bfloat16))
        for k in ("dX", "dW1", "dW3", "dW2"):
            getattr(grads, k).fill_(float("nan"))
        graph.replay()
        call(ref_grads, ref_ws)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        for k in ("dX", "dW1", "dW3", "dW2"):
            assert torch.equal(getattr(grads, k), getattr(ref_grads, k)), (i, k)


def test_dense_ffn_backward_replays_as_a_graph(s3r):
    T, d, F, S = 2048, 512, 1536, 1024
    inp = workloads.ffn_inputs(T, d, F, S, seed=41)
    c = lambda t: t.cuda()
    ops = s3r.ffn_forward_operands(c(inp.X), c(inp.W1), c(inp.W3), c(inp.W2), c(inp.a), c(inp.h1), c(inp.h3))
    _check_capture(s3r, ops, c(inp.dY), S, None)


def test_grouped_ffn_backward_replays_as_a_graph(s3r):
    d, F = 256, 384
    mi = workloads.moe_inputs_sized([700, 0, 129, 1024, 64, 300], d, F, seed=43)
    c = lambda t: t.cuda()
    ops = s3r.moe_forward_operands(c(mi.X), c(mi.W1), c(mi.W3), c(mi.W2), c(mi.a), c(mi.h1), c(mi.h3))
    _check_capture(s3r, ops, c(mi.dY), 0, list(mi.offsets))
