"""GPU parity: the tile quantizers against the CPU oracle.

Codes and tile scales bit-exact; error partial sums within the fp32 bound.
Covers ragged tiles, unaligned row strides, the folds, all three rounding
modes, the full-size quantize sweep (sampled windows) and the device status.
"""
import numpy as np
import pytest
import torch

import workloads
from parity_util import assert_close_mag, codes

pytestmark = pytest.mark.gpu

MODES = ["S3R", "INDEP", "RTNE"]


@pytest.fixture(scope="module")
def s3r():
    import stochastic_rounding_int8_gb300 as m
    m.lib()
    return m


def _gpu_quant(s3r, mode, G, s_x, s_w, seed, tid, fmt=1):
    if mode == "S3R":
        o = s3r.s3r_quantize(G, s_x, s_w, seed, tid, code_format=fmt)
        return o.Q, o.tile_scale, o.tok_err_part, o.col_err_part
    if mode == "INDEP":
        o = s3r.indep_sr_quantize(G, s_x, s_w, seed, tid, code_format=fmt)
        return o.Q, o.tile_scale, None, None
    Q, sc = s3r.rtne_quantize(G, s3r.AXIS_TILE, s_x=s_x, s_w=s_w, code_format=fmt)
    return Q, sc, None, None


def _case(T, N, seed, ld=None, outliers=False):
    rng = np.random.default_rng(seed)
    g = rng.standard_t(3, size=(T, N)).astype(np.float32) * np.float32(1e-3)
    if outliers:
        g = np.where(rng.random((T, N)) < 0.01, g * 100, g).astype(np.float32)
    Gb = torch.from_numpy(g).to(torch.bfloat16)
    if ld is not None and ld != N:
        big = torch.zeros((T, ld), dtype=torch.bfloat16)
        big[:, :N] = Gb
        Gb = big[:, :N]
    s_x = torch.from_numpy((rng.random(T) * 0.05 + 0.01).astype(np.float32))
    s_w = torch.from_numpy((rng.random(N) * 1e-3 + 1e-4).astype(np.float32))
    return Gb, s_x, s_w


@pytest.mark.parametrize("fmt", [0, 1], ids=["s8", "f16"])
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("T,N,ld,fold", [(256, 1024, None, True), (300, 260, None, True), (1, 8, None, False),
                                         (129, 136, None, True), (200, 1001, 1001, True), (130, 96, 128, False),
                                         (513, 384, None, True)])
def test_quantize_parity(s3r, orc, fmt, mode, T, N, ld, fold):
    Gb, s_x, s_w = _case(T, N, T * 7 + N, ld)
    dev = "cuda"
    Gd = Gb.to(dev) if ld is None else torch.zeros((T, ld), dtype=torch.bfloat16, device=dev)[:, :N].copy_(Gb.to(dev))
    sxd, swd = (s_x.to(dev), s_w.to(dev)) if fold else (None, None)
    seed, tid = 1234567, 5
    Q, sc, tok, col = _gpu_quant(s3r, mode, Gd, sxd, swd, seed, tid, fmt)
    torch.cuda.synchronize()
    G = orc.from_torch_bf16(Gb.contiguous())
    Qo, do, Eo, st = orc.quantize(G, s_x.numpy() if fold else None, s_w.numpy() if fold else None,
                                  mode=getattr(orc, mode), seed=seed, tensor_id=tid)
    assert st == 0
    Qg = codes(Q)
    assert np.array_equal(Qg, Qo), f"codes differ in {(Qg != Qo).sum()} elements"
    assert np.array_equal(sc.cpu().numpy(), do)
    if tok is not None:
        tok_o, col_o = orc.error_partials(Eo)
        tok_m, col_m = orc.error_partials(np.abs(Eo))
        assert_close_mag(tok.cpu().numpy(), tok_o, tok_m, "tok_err_part")
        assert_close_mag(col.cpu().numpy(), col_o, col_m, "col_err_part")


@pytest.mark.parametrize("T", [4096, 16384, 65536])
def test_quantize_sweep_full_size_sampled(s3r, orc, T):
    """The quantize-only sweep at N = 8192: full GPU pass, oracle on sampled
    tile-aligned windows (thresholds at their global indices)."""
    N = 8192
    Gb = workloads.quantize_sweep_input(T, N, seed=workloads.DATA_SEED + 3)
    Gd = Gb.cuda()
    rng = np.random.default_rng(T)
    windows = [(0, 0), ((T // 128 - 1) * 128, N - 512)]
    windows += [(int(rng.integers(0, T // 128)) * 128, int(rng.integers(0, N // 128 - 4)) * 128) for _ in range(2)]
    for mode in MODES:
        Q, sc, tok, col = _gpu_quant(s3r, mode, Gd, None, None, 77, 3, fmt=(T // 4096) % 2)
        Q, sc = codes(Q), sc.cpu().numpy()
        tok = tok.cpu().numpy() if tok is not None else None
        for (r0, c0) in windows:
            Gw = orc.from_torch_bf16(Gb[r0:r0 + 128, c0:c0 + 512].contiguous())
            Qo, do, Eo, _ = orc.quantize(Gw, mode=getattr(orc, mode), seed=77, tensor_id=3, window=(r0, c0, N))
            assert np.array_equal(Q[r0:r0 + 128, c0:c0 + 512], Qo), (mode, r0, c0)
            assert np.array_equal(sc[r0 // 128, c0 // 128:c0 // 128 + 4], do[0])
            if tok is not None:
                t_o, _ = orc.error_partials(Eo)
                t_m, _ = orc.error_partials(np.abs(Eo))
                assert_close_mag(tok[r0:r0 + 128, c0 // 128:c0 // 128 + 4], t_o, t_m, "tok window")


def test_quantize_deterministic_and_seed_sensitive(s3r):
    Gb, s_x, s_w = _case(384, 512, 9)
    G = Gb.cuda()
    a = s3r.s3r_quantize(G, seed=1, tensor_id=0).Q.clone()
    a8 = s3r.s3r_quantize(G, seed=1, tensor_id=0, code_format=s3r.CODES_S8).Q
    assert np.array_equal(codes(a), codes(a8))
    b = s3r.s3r_quantize(G, seed=1, tensor_id=0).Q
    c = s3r.s3r_quantize(G, seed=2, tensor_id=0).Q
    d = s3r.s3r_quantize(G, seed=1, tensor_id=1).Q
    assert torch.equal(a, b)
    assert not torch.equal(a, c) and not torch.equal(a, d)


def test_nonfinite_sets_device_status(s3r):
    Gb, _, _ = _case(256, 256, 10)
    Gb[3, 200] = float("nan")
    st = s3r.new_status()
    o = s3r.s3r_quantize(Gb.cuda(), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == -4
    sc = o.tile_scale.cpu()
    assert torch.isnan(sc[0, 1]) and torch.isfinite(sc[0, 0]) and torch.isfinite(sc[1]).all()
    assert not codes(o.Q)[:128, 128:].any()
    with pytest.raises(s3r.S3RError):
        s3r.check_status(st)


def test_zero_tile(s3r):
    G = torch.zeros((200, 300), dtype=torch.bfloat16, device="cuda")
    G[150, 290] = 1.0
    o = s3r.s3r_quantize(G)
    sc = o.tile_scale.cpu()
    assert sc[0, 0] == 0 and sc[1, 2] == np.float32(1.0) / np.float32(127.0)
    q = codes(o.Q).astype(np.int64)
    assert q[150, 290] == 127 and np.abs(q).sum() == 127
    tok = o.tok_err_part.cpu().numpy()
    # all-zero tiles carry no error; the lone element's error is Delta*127 - 1 (Delta is rounded)
    want = np.float32(np.float32(1.0) / np.float32(127.0)) * np.float64(127.0) - 1.0
    assert tok[150, 2] == np.float32(want)
    tok[150, 2] = 0.0
    assert not tok.any() and float(o.col_err_part.cpu()[0].abs().sum()) == 0.0


@pytest.mark.parametrize("fmt", [0, 1], ids=["s8", "f16"])
@pytest.mark.parametrize("mode,S", [("S3R_7BIT", 0), ("BCAST", 0), ("BCAST", 128), ("BCAST", 256)])
@pytest.mark.parametrize("T,N,fold", [(256, 1024, True), (300, 260, False), (512, 384, True), (129, 136, True)])
def test_paper_modes_parity(s3r, orc, fmt, mode, S, T, N, fold):
    """The paper's 7-bit thresholds and the per-example Phi_bcast: codes and
    tile scales bit for bit, error partials within the fp32 bound."""
    if S and T % S:
        pytest.skip("examples must tile the rows")
    Gb, s_x, s_w = _case(T, N, T * 5 + N + S)
    sxd, swd = (s_x.cuda(), s_w.cuda()) if fold else (None, None)
    seed, tid = 77, 9
    o, amax = s3r.s3r_quantize_ex(Gb.cuda(), sxd, swd, getattr(s3r, "ROUND_" + mode), S, seed=seed, tensor_id=tid,
                                  code_format=fmt)
    torch.cuda.synchronize()
    assert amax is None
    G = orc.from_torch_bf16(Gb)
    omode = orc.S3R7 if mode == "S3R_7BIT" else orc.BCAST
    Qo, do, Eo, st = orc.quantize(G, s_x.numpy() if fold else None, s_w.numpy() if fold else None, mode=omode,
                                  seed=seed, tensor_id=tid, S=S)
    assert st == 0
    assert np.array_equal(codes(o.Q), Qo), f"codes differ in {(codes(o.Q) != Qo).sum()} elements"
    assert np.array_equal(o.tile_scale.cpu().numpy(), do)
    tok_o, col_o = orc.error_partials(Eo)
    tok_m, col_m = orc.error_partials(np.abs(Eo))
    assert_close_mag(o.tok_err_part.cpu().numpy(), tok_o, tok_m, "tok_err_part")
    assert_close_mag(o.col_err_part.cpu().numpy(), col_o, col_m, "col_err_part")


@pytest.mark.parametrize("fmt", [0, 1], ids=["s8", "f16"])
@pytest.mark.parametrize("mode", ["S3R", "S3R_7BIT", "RTNE"])
@pytest.mark.parametrize("T,N", [(384, 512), (300, 260)])
def test_per_tensor_step_parity(s3r, orc, fmt, mode, T, N):
    """[S3R]'s per-tensor step: one Delta = max|G'|/127 for every tile, codes
    bit for bit against the oracle with one tile covering the tensor."""
    Gb, s_x, s_w = _case(T, N, T + 3 * N, outliers=True)
    o, amax = s3r.s3r_quantize_ex(Gb.cuda(), s_x.cuda(), s_w.cuda(), getattr(s3r, "ROUND_" + mode), 0,
                                  per_tensor=True, seed=3, tensor_id=1, code_format=fmt)
    torch.cuda.synchronize()
    G = orc.from_torch_bf16(Gb)
    omode = {"S3R": orc.S3R, "S3R_7BIT": orc.S3R7, "RTNE": orc.RTNE}[mode]
    Qo, do, Eo, _ = orc.quantize(G, s_x.numpy(), s_w.numpy(), mode=omode, seed=3, tensor_id=1, tile=(T, N))
    g = ((s_x.numpy()[:, None] * G).astype(np.float32) * s_w.numpy()[None, :]).astype(np.float32)
    assert amax.item() == np.abs(g).max()
    assert np.array_equal(codes(o.Q), Qo)
    assert np.all(o.tile_scale.cpu().numpy() == do[0, 0])
    if mode != "RTNE":
        tok_o, col_o = orc.error_partials(Eo)
        tok_m, col_m = orc.error_partials(np.abs(Eo))
        assert_close_mag(o.tok_err_part.cpu().numpy(), tok_o, tok_m, "tok_err_part")
        assert_close_mag(o.col_err_part.cpu().numpy(), col_o, col_m, "col_err_part")
