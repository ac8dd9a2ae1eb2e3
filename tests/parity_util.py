"""Comparison helpers shared by the GPU parity tests.

Tolerances.  Integer results (codes, int32 block partials, row sums) must be
bit-exact.  fp32 results are compared against the fp64 oracle with
|gpu - ref| <= RTOL * mag + ATOL_REL * max(mag), where mag is the sum of the
absolute values of the terms that make up each result (the natural bound of a
reordered fp32 sum: n * 2^-24 * sum|terms| with n up to ~112 blocks stays
below 1e-5 * sum|terms|).  RTOL = 1e-5 is the stated relative tolerance; the
stated absolute 1e-6 is applied relative to the tensor's magnitude because the
gradients here are ~1e-8..1e-3 in absolute value.
"""
from __future__ import annotations

import numpy as np

RTOL = 1e-5
ATOL_REL = 1e-6
TILE = 128


def codes(Q):
    """Device code tensor (int8 or float16 holding integers) -> int8 numpy."""
    import torch
    q = Q.detach().cpu()
    if q.dtype == torch.float16:
        f = q.float()
        assert torch.equal(f, f.round()) and float(f.abs().max()) <= 127, "fp16 codes must be integers in [-127, 127]"
        q = f.to(torch.int8)
    return q.numpy()


def assert_close_mag(got, ref, mag, what, rtol=RTOL, atol_rel=ATOL_REL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    mag = np.asarray(mag, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    tol = rtol * mag + atol_rel * (float(mag.max()) if mag.size else 0.0) + 1e-30
    err = np.abs(got - ref)
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err / tol), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r} tol {tol[i]!r}")


def expand_tiles(delta, T, N, tr=TILE, tc=TILE):
    return np.repeat(np.repeat(np.asarray(delta, dtype=np.float64), tr, 0), tc, 1)[:T, :N]


def _mm(a, b):
    """float64 matrix product (torch's CPU matmul: multi-threaded)."""
    import torch
    return (torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64)) @
            torch.from_numpy(np.ascontiguousarray(b, dtype=np.float64))).numpy()


def dx_magnitude(Q, delta, W8, s_x, eps=None, rowsum=None, v=None, S=None, rows=None):
    """sum_kb |delta| * |sum_n Q W8| bounded above by |Delta Q| |W8|^T, plus the
    correction terms, over |s_x|: an upper bound of the terms' absolute sum."""
    T, N = Q.shape
    rows = np.arange(T) if rows is None else np.asarray(rows)
    G = np.abs(expand_tiles(delta, T, N)[rows] * Q[rows].astype(np.float64))
    mag = _mm(G, np.abs(W8.astype(np.float64)).T)
    if eps is not None:
        mag = mag + np.abs(eps[rows])[:, None] * np.abs(rowsum.astype(np.float64))[None, :]
        mag = mag + np.abs(v[rows // S])
    sx = np.ones(len(rows)) if s_x is None else np.abs(np.asarray(s_x, dtype=np.float64)[rows])
    return mag / sx[:, None]


def dw_magnitude(X8, Q, delta, s_w, colmean=None, mu=None, xsum=None, p=None, krows=None):
    T, K = X8.shape
    N = Q.shape[1]
    krows = np.arange(K) if krows is None else np.asarray(krows)
    G = np.abs(expand_tiles(delta, T, N) * Q.astype(np.float64))
    mag = _mm(np.abs(X8[:, krows].astype(np.float64)).T, G)
    if colmean is not None:
        cm = np.abs(colmean - mu[:, None])
        mag = mag + np.abs(xsum[:, krows].astype(np.float64)).T @ cm + np.abs(p[krows])[:, None]
    sw = np.ones(N) if s_w is None else np.abs(np.asarray(s_w, dtype=np.float64))
    return mag / sw[None, :]


def projection(D, S):
    """Orthogonal projection of each example's block of D onto row- and
    column-constant matrices (the same subspace as the correction)."""
    T, N = D.shape
    out = np.empty_like(D, dtype=np.float64)
    for b in range(T // S):
        blk = D[b * S:(b + 1) * S].astype(np.float64)
        out[b * S:(b + 1) * S] = blk.mean(1, keepdims=True) + blk.mean(0, keepdims=True) - blk.mean()
    return out


def near_tie_flips(Q_gpu, Q_orc, y_orc, u, max_frac=1e-3, margin=1e-3):
    """Codes may differ only by one step and only where the oracle's own
    decision was within `margin` of flipping (threshold vs residual, or y
    next to an integer).  u: thresholds broadcastable to y ([T, 1] per token,
    [T, N] per element, 0.5 for round-to-nearest).  Returns the mismatch mask."""
    diff = Q_gpu.astype(np.int32) - Q_orc.astype(np.int32)
    mask = diff != 0
    if not mask.any():
        return mask
    assert np.abs(diff[mask]).max() == 1, "codes differ by more than one step"
    assert mask.mean() <= max_frac, f"too many code flips: {mask.mean():.2e}"
    f = np.floor(y_orc)
    p = y_orc - f
    close = np.minimum(np.abs(p - u), np.minimum(p, 1 - p)) < margin
    assert close[mask].all(), "a code differs where the oracle's decision was not a near tie"
    return mask


def tile_amax(g, tile=TILE):
    """Per-128x128-tile absmax of g [T, N] (ragged edges included), float32."""
    T, N = g.shape
    nt, nn = -(-T // tile), -(-N // tile)
    pad = np.zeros((nt * tile, nn * tile), dtype=np.float32)
    pad[:T, :N] = np.abs(g)
    return pad.reshape(nt, tile, nn, tile).max(axis=(1, 3))


def flip_effect(Qg, dg, Qo, do, W8, X8, s_x, s_w, S, dx_ec, dw_ec, rows, krows, chunk=2048):
    """Exact change of dX[rows] and dW[krows] of one linear when the oracle's
    dequantized gradient Delta_o Q_o is replaced by Delta_g Q_g, i.e. by
    D = Delta_g Q_g - Delta_o Q_o: through the correction (D - P(D), P the
    per-example projection onto row- and column-constant matrices) where the
    mode applies it, then both products and the rescales.  Streams D in
    chunks of rows, so it never holds the whole [T, N] difference."""
    T, N = Qg.shape
    assert chunk % TILE == 0
    rows = np.asarray(rows, dtype=np.int64)
    krows = np.asarray(krows, dtype=np.int64)
    B = T // S
    rowsum = np.zeros(T)
    colsum = np.zeros((B, N))
    XD = np.zeros((krows.size, N))
    Drows = np.zeros((rows.size, N))
    pos = {int(r): i for i, r in enumerate(rows)}
    X8k = X8[:, krows].astype(np.float64)
    for t0 in range(0, T, chunk):
        t1 = min(T, t0 + chunk)
        tr = t0 // TILE   # chunk is a multiple of the tile height
        Dc = (expand_tiles(dg[tr:], t1 - t0, N) * Qg[t0:t1].astype(np.float64)
              - expand_tiles(do[tr:], t1 - t0, N) * Qo[t0:t1].astype(np.float64))
        rowsum[t0:t1] = Dc.sum(1)
        for b in range(t0 // S, (t1 - 1) // S + 1):
            a0, a1 = max(t0, b * S), min(t1, (b + 1) * S)
            colsum[b] += Dc[a0 - t0:a1 - t0].sum(0)
        XD += _mm(X8k[t0:t1].T, Dc)
        sel = rows[(rows >= t0) & (rows < t1)]
        for r in sel:
            Drows[pos[int(r)]] = Dc[r - t0]
    rowmean = rowsum / N
    colmean = colsum / S
    mu = rowsum.reshape(B, S).sum(1) / (S * N)
    b_of = rows // S
    if dx_ec:
        Drows = Drows - rowmean[rows][:, None] - colmean[b_of] + mu[b_of][:, None]
    ddx = _mm(Drows, W8.astype(np.float64).T) / np.asarray(s_x, dtype=np.float64)[rows][:, None]
    if dw_ec:
        xs = X8k.reshape(B, S, krows.size).sum(1)                  # [B, nk]
        XD = XD - (X8k.T @ rowmean)[:, None] - xs.T @ colmean + (xs.T @ mu)[:, None]
    ddw = XD / np.asarray(s_w, dtype=np.float64)[None, :]
    return ddx, ddw
