"""The allocation-free correction entry point (s3r_ec_correct_static).

Callers that cannot allocate device memory while they run the backward --
host callbacks and real-time loops, where an allocation may block or fail,
and deployments with a device budget fixed up front -- use this variant,
whose scratch lives in a static array of the library instead of a caller
workspace.  The test calls it through the C ABI twice in a row (two different
gradients, so the second call runs over the first call's leftover scratch)
and checks each result against s3r_ec_correct with a torch-allocated
workspace.  Both run the same kernels over the same inputs, and every sum in
them has a fixed order (chunk partials and per-example means are added in
index order, never by atomics), so the results must match bit for bit: a
counter or a partial left over from the first call would show as a
difference.  This file is collected last on purpose.
"""
import ctypes as C

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _outputs(T, N, K, S, dev):
    B = T // S
    f = lambda *s: torch.full(s, float("nan"), dtype=torch.float32, device=dev)
    i = lambda *s: torch.full(s, -7, dtype=torch.int32, device=dev)
    return dict(eps=f(T), mu=f(B), colmean=f(B, N), rowsum=i(K), v=f(B, K), xsum=i(B, K), p=f(K))


def _call(L, fn, q, T, N, S, W, X, fmt, out, ws=None, status=None):
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = [_ptr(q.tok_err_part), _ptr(q.col_err_part), T, N, S, _ptr(W), W.shape[0], _ptr(X), fmt, 2,
            _ptr(out["eps"]), _ptr(out["mu"]), _ptr(out["colmean"]), _ptr(out["rowsum"]), _ptr(out["v"]),
            _ptr(out["xsum"]), _ptr(out["p"])]
    if fn == "s3r_ec_correct":
        args += [_ptr(ws), ws.numel()]
    args += [_ptr(status), stream]
    return getattr(L, fn)(*args)


@pytest.mark.parametrize("fmt", [0, 1], ids=["s8", "f16"])
def test_static_scratch_matches_workspace_version_twice(fmt):
    import stochastic_rounding_int8_gb300 as s3r
    L = s3r.lib()
    T, N, K, S = 8192, 2048, 5632, 2048      # the W2 linear of the d=2048, F=5632 FFN block
    dev = "cuda"
    rng = np.random.default_rng(99)
    dt = torch.float16 if fmt else torch.int8
    W = torch.from_numpy(rng.integers(-127, 128, size=(K, N)).astype(np.int8)).to(dt).to(dev)
    X = torch.from_numpy(rng.integers(-127, 128, size=(T, K)).astype(np.int8)).to(dt).to(dev)
    st = s3r.new_status()
    for call in range(2):
        G = torch.from_numpy((rng.standard_t(3, size=(T, N)) * 1e-3).astype(np.float32)).to(torch.bfloat16).to(dev)
        q = s3r.s3r_quantize(G, seed=call, tensor_id=3, code_format=fmt)
        ref = _outputs(T, N, K, S, dev)
        ws = torch.empty(L.s3r_ec_workspace_size(T, K), dtype=torch.uint8, device=dev)
        assert _call(L, "s3r_ec_correct", q, T, N, S, W, X, fmt, ref, ws=ws) == 0
        got = _outputs(T, N, K, S, dev)
        assert _call(L, "s3r_ec_correct_static", q, T, N, S, W, X, fmt, got, status=st) == 0, \
            L.s3r_last_error().decode()
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        for k in ("rowsum", "xsum", "eps", "mu", "colmean", "v", "p"):
            assert torch.equal(got[k], ref[k]), (call, k)


def test_static_scratch_rejects_oversized_problem():
    import stochastic_rounding_int8_gb300 as s3r
    L = s3r.lib()
    T, N, K, S = 16384, 256, 16384, 16384    # needs 128 chunks x 16384 x 8 B = 16 MiB of scratch
    dev = "cuda"
    q = s3r.s3r_quantize(torch.zeros((T, N), dtype=torch.bfloat16, device=dev))
    W = torch.zeros((K, N), dtype=torch.float16, device=dev)
    X = torch.zeros((T, K), dtype=torch.float16, device=dev)
    out = _outputs(T, N, K, S, dev)
    assert _call(L, "s3r_ec_correct_static", q, T, N, S, W, X, 1, out) == -8
    assert "static array holds" in L.s3r_last_error().decode()


@pytest.mark.parametrize("fmt", [0, 1], ids=["s8", "f16"])
def test_static_scratch_in_a_captured_graph(fmt):
    """The call inside a CUDA graph capture (the global capture mode, which
    refuses calls that could allocate or synchronize), then replayed over new
    gradients written into the captured partials: every replay must equal the
    workspace version on the same inputs bit for bit."""
    import stochastic_rounding_int8_gb300 as s3r
    L = s3r.lib()
    T, N, K, S = 4096, 1024, 2816, 1024
    dev = "cuda"
    rng = np.random.default_rng(7)
    dt = torch.float16 if fmt else torch.int8
    W = torch.from_numpy(rng.integers(-127, 128, size=(K, N)).astype(np.int8)).to(dt).to(dev)
    X = torch.from_numpy(rng.integers(-127, 128, size=(T, K)).astype(np.int8)).to(dt).to(dev)
    grad = lambda: torch.from_numpy((rng.standard_t(3, size=(T, N)) * 1e-3).astype(np.float32)).to(
        torch.bfloat16).to(dev)
    q = s3r.s3r_quantize(grad(), seed=0, tensor_id=3, code_format=fmt)
    st = s3r.new_status()
    got = _outputs(T, N, K, S, dev)
    assert _call(L, "s3r_ec_correct_static", q, T, N, S, W, X, fmt, got, status=st) == 0   # warm-up, eager
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        rc = _call(L, "s3r_ec_correct_static", q, T, N, S, W, X, fmt, got, status=st)
    assert rc == 0, L.s3r_last_error().decode()
    ws = torch.empty(L.s3r_ec_workspace_size(T, K), dtype=torch.uint8, device=dev)
    for rep in range(3):
        s3r.s3r_quantize(grad(), seed=10 + rep, tensor_id=3, code_format=fmt, out=q)
        for v in got.values():
            v.fill_(-1)
        g.replay()
        ref = _outputs(T, N, K, S, dev)
        assert _call(L, "s3r_ec_correct", q, T, N, S, W, X, fmt, ref, ws=ws) == 0
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        for k in ("rowsum", "xsum", "eps", "mu", "colmean", "v", "p"):
            assert torch.equal(got[k], ref[k]), (rep, k)
