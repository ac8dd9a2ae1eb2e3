"""CPU oracle for the S3R / S3R-EC INT8 backward -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The CUDA library never calls it and shares no code
with it.  The arithmetic lives in ``s3r_oracle.c`` (plain single-threaded C);
this module builds it with gcc, loads it with ctypes, and composes its pieces
into the linear-layer and SwiGLU-FFN backward passes step by step, in the order
of the S3R paper ("Efficient Quantization Training with Stochastic Rounding via
Structured Subspace Randomness", §III-A to §III-D).

Parity pins: every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_*.py`` (worked example, closed forms, invariants, library
routines, brute force).  Whole-pipeline training quality (the paper's Tables I
and II) is *parity unpinned*: it needs the C4 data set and trained checkpoints.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "s3r_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liborc_s3r.so")
_lock = threading.Lock()
_lib = None

RTNE, S3R, INDEP, S3R7, BCAST = 0, 1, 2, 3, 4
EC_NONE, EC_DX_ONLY, EC_TWO_WAY, EC_DX_TOKEN_ONLY, EC_DW_ONLY = 0, 1, 2, 3, 4
SHARED = (S3R, S3R7, BCAST)   # modes with one threshold tensor for both products
TILE = 128


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fused multiply-add contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                               "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = C.CDLL(build())
            L = _lib
            L.orc_word_to_unit.restype = C.c_float
            L.orc_word_to_unit.argtypes = [C.c_uint32]
            L.orc_token_threshold.restype = C.c_float
            L.orc_token_threshold.argtypes = [C.c_uint64, C.c_uint64, C.c_uint32]
            L.orc_element_threshold.restype = C.c_float
            L.orc_element_threshold.argtypes = [C.c_uint64, C.c_uint64, C.c_uint32]
            L.orc_token_threshold7.restype = C.c_float
            L.orc_token_threshold7.argtypes = [C.c_uint64, C.c_uint64, C.c_uint32]
            L.orc_example_threshold.restype = C.c_float
            L.orc_example_threshold.argtypes = [C.c_uint64, C.c_uint64, C.c_uint32]
            L.orc_quantize_window_ex.restype = C.c_int
            L.orc_float_to_bf16.restype = C.c_uint16
            L.orc_float_to_bf16.argtypes = [C.c_float]
            L.orc_sr_bf16.restype = C.c_uint16
            L.orc_sr_bf16.argtypes = [C.c_float, C.c_uint32]
            L.orc_sr_bf16_matrix.restype = C.c_int
            L.orc_sr_e4m3.restype = C.c_uint8
            L.orc_sr_e4m3.argtypes = [C.c_float, C.c_uint32]
            L.orc_rn_e4m3.restype = C.c_uint8
            L.orc_rn_e4m3.argtypes = [C.c_float]
            L.orc_sr_fp8_matrix.restype = C.c_int
            L.orc_inv127_rz.restype = C.c_float
            L.orc_inv127_rz.argtypes = [C.c_float]
            L.orc_sr_step.restype = C.c_float
            L.orc_sr_step.argtypes = [C.c_float, C.c_float]
            L.orc_expf.restype = C.c_float
            L.orc_expf.argtypes = [C.c_float]
            L.orc_sigmoidf.restype = C.c_float
            L.orc_sigmoidf.argtypes = [C.c_float]
            L.orc_quantize.restype = C.c_int
            L.orc_quantize_window.restype = C.c_int
            L.orc_rtne_operand.restype = C.c_int
            L.orc_error_stats.restype = C.c_int
        return _lib


def _p(a):
    return None if a is None else C.c_void_p(a.ctypes.data)


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def _i64(x):
    return C.c_int64(int(x))


# --------------------------------------------------------------------------
# primitives
# --------------------------------------------------------------------------
def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def word_to_unit(w: int) -> float:
    return lib().orc_word_to_unit(int(w) & 0xFFFFFFFF)


def token_threshold(t: int, seed: int, tensor_id: int) -> float:
    return lib().orc_token_threshold(int(t), int(seed), int(tensor_id))


def token_threshold7(t: int, seed: int, tensor_id: int) -> float:
    """[S3R] §III-B: 7-bit threshold of token t (byte t mod 4 of the word of t / 4, half-step shift)."""
    return lib().orc_token_threshold7(int(t), int(seed), int(tensor_id))


def example_threshold(b: int, seed: int, tensor_id: int) -> float:
    """[S3R] §III-B, Phi_bcast: the threshold shared by every element of example b."""
    return lib().orc_example_threshold(int(b), int(seed), int(tensor_id))


def element_threshold(e: int, seed: int, tensor_id: int) -> float:
    return lib().orc_element_threshold(int(e), int(seed), int(tensor_id))


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32, exactly."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float32)
    lib().orc_bf16_array_to_float(_p(b), _i64(b.size), _p(out))
    return out


def from_torch_bf16(t) -> np.ndarray:
    """A torch bf16 CPU tensor -> float32 numpy, via the oracle's own widening."""
    import torch
    return bf16_to_f32(t.contiguous().view(torch.int16).numpy().view(np.uint16))


def inv127_rz(a: float) -> float:
    """127 / a rounded toward zero (the quantizer's normalizing factor)."""
    return lib().orc_inv127_rz(float(a))


def sr_step(y: float, u: float) -> float:
    """One stochastic rounding of y to the unit grid with threshold u."""
    return lib().orc_sr_step(float(y), float(u))


def expf(x: float) -> float:
    return lib().orc_expf(float(x))


def sigmoidf(x: float) -> float:
    return lib().orc_sigmoidf(float(x))


def quantize(G, s_x=None, s_w=None, mode=S3R, seed=0, tensor_id=0, tile=(TILE, TILE), window=None, S=0):
    """Fold, tile-scale and round G (float32 [T, N]).

    window = (row_base, col_base, n_global) treats G as a tile-aligned window
    of a larger tensor (thresholds use global indices).  S: tokens per example
    (Phi_bcast; 0 = one example).  tile=(T, N) gives the paper's per-tensor step.
    Returns (Q int8 [T,N], delta f32 [ceil(T/tr), ceil(N/tc)], E f32 [T,N], status)."""
    G = _f32(G)
    T, N = G.shape
    tr, tc = tile
    ntr, ntc = -(-T // tr), -(-N // tc)
    Q = np.zeros((T, N), dtype=np.int8)
    delta = np.zeros((ntr, ntc), dtype=np.float32)
    E = np.zeros((T, N), dtype=np.float32)
    rb, cb, ng = window if window is not None else (0, 0, N)
    st = lib().orc_quantize_window_ex(_p(G), _i64(T), _i64(N), _i64(N), _p(_f32(s_x)), _p(_f32(s_w)),
                                      C.c_int(mode), _i64(S), C.c_uint64(seed), C.c_uint32(tensor_id), _i64(tr),
                                      _i64(tc), _p(Q), _p(delta), _p(E), _i64(rb), _i64(cb), _i64(ng))
    return Q, delta, E, st


def rtne_operand(A, axis: int):
    """Forward RTNE operand with a per-row (axis 0) or per-column (axis 1) scale."""
    A = _f32(A)
    R, Cc = A.shape
    Q = np.zeros((R, Cc), dtype=np.int8)
    scale = np.zeros(R if axis == 0 else Cc, dtype=np.float32)
    st = lib().orc_rtne_operand(_p(A), _i64(R), _i64(Cc), _i64(Cc), C.c_int(axis), _p(Q), _p(scale))
    if st != 0:
        raise ValueError(f"orc_rtne_operand status {st}")
    return Q, scale


def error_partials(E, tile=(TILE, TILE)):
    E = _f32(E)
    T, N = E.shape
    tr, tc = tile
    tok = np.zeros((T, -(-N // tc)), dtype=np.float64)
    col = np.zeros((-(-T // tr), N), dtype=np.float64)
    lib().orc_error_partials(_p(E), _i64(T), _i64(N), _i64(tr), _i64(tc), _p(tok), _p(col))
    return tok, col


def error_stats(E, S: int):
    E = _f32(E)
    T, N = E.shape
    B = T // S
    eps = np.zeros(T, dtype=np.float64)
    colmean = np.zeros((B, N), dtype=np.float64)
    mu = np.zeros(B, dtype=np.float64)
    st = lib().orc_error_stats(_p(E), _i64(T), _i64(N), _i64(S), _p(eps), _p(colmean), _p(mu))
    if st != 0:
        raise ValueError("T must be a multiple of S")
    return eps, colmean, mu


def ec_factors(eps, colmean, mu, S: int, W8, X8=None):
    W8 = np.ascontiguousarray(W8, dtype=np.int8)
    K, N = W8.shape
    T = eps.shape[0]
    B = T // S
    rowsum = np.zeros(K, dtype=np.int64)
    v = np.zeros((B, K), dtype=np.float64)
    xsum = np.zeros((B, K), dtype=np.int64)
    p = np.zeros(K, dtype=np.float64)
    X8c = None if X8 is None else np.ascontiguousarray(X8, dtype=np.int8)
    lib().orc_ec_factors(_p(np.ascontiguousarray(eps, dtype=np.float64)),
                         _p(np.ascontiguousarray(colmean, dtype=np.float64)),
                         _p(np.ascontiguousarray(mu, dtype=np.float64)),
                         _i64(T), _i64(N), _i64(S), _p(W8), _p(X8c), _i64(K), _p(rowsum), _p(v), _p(xsum), _p(p))
    return rowsum, v, xsum, p


def dx_blocks(Q, W8, rows, blk=TILE):
    Q = np.ascontiguousarray(Q, dtype=np.int8)
    W8 = np.ascontiguousarray(W8, dtype=np.int8)
    T, N = Q.shape
    K = W8.shape[0]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    nkb = -(-N // blk)
    out = np.zeros((rows.size, K, nkb), dtype=np.int32)
    lib().orc_dx_blocks(_p(Q), _p(W8), _i64(T), _i64(N), _i64(K), _i64(blk), _p(rows), _i64(rows.size), _p(out))
    return out


def dw_blocks(X8, Q, krows, blk=TILE):
    X8 = np.ascontiguousarray(X8, dtype=np.int8)
    Q = np.ascontiguousarray(Q, dtype=np.int8)
    T, K = X8.shape
    N = Q.shape[1]
    krows = np.ascontiguousarray(krows, dtype=np.int64)
    ntb = -(-T // blk)
    out = np.zeros((krows.size, N, ntb), dtype=np.int32)
    lib().orc_dw_blocks(_p(X8), _p(Q), _i64(T), _i64(K), _i64(N), _i64(blk), _p(krows), _i64(krows.size), _p(out))
    return out


def dx(Q, delta, W8, s_x, ec_mode, eps, rowsum, v, S, rows, tile=(TILE, TILE)):
    Q = np.ascontiguousarray(Q, dtype=np.int8)
    W8 = np.ascontiguousarray(W8, dtype=np.int8)
    T, N = Q.shape
    K = W8.shape[0]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.zeros((rows.size, K), dtype=np.float64)
    f64 = lambda a: None if a is None else np.ascontiguousarray(a, dtype=np.float64)
    i64 = lambda a: None if a is None else np.ascontiguousarray(a, dtype=np.int64)
    lib().orc_dx(_p(Q), _p(_f32(delta)), _p(W8), _i64(T), _i64(N), _i64(K), _i64(tile[0]), _i64(tile[1]),
                 _p(_f32(s_x)), C.c_int(ec_mode), _p(f64(eps)), _p(i64(rowsum)), _p(f64(v)), _i64(S),
                 _p(rows), _i64(rows.size), _p(out))
    return out


def dw(X8, Q, delta, s_w, ec_mode, colmean, mu, xsum, p, S, krows, tile=(TILE, TILE)):
    X8 = np.ascontiguousarray(X8, dtype=np.int8)
    Q = np.ascontiguousarray(Q, dtype=np.int8)
    T, K = X8.shape
    N = Q.shape[1]
    krows = np.ascontiguousarray(krows, dtype=np.int64)
    out = np.zeros((krows.size, N), dtype=np.float64)
    f64 = lambda a: None if a is None else np.ascontiguousarray(a, dtype=np.float64)
    i64 = lambda a: None if a is None else np.ascontiguousarray(a, dtype=np.int64)
    lib().orc_dw(_p(X8), _p(Q), _p(_f32(delta)), _i64(T), _i64(K), _i64(N), _i64(tile[0]), _i64(tile[1]),
                 _p(_f32(s_w)), C.c_int(ec_mode), _p(f64(colmean)), _p(f64(mu)), _p(i64(xsum)), _p(f64(p)), _i64(S),
                 _p(krows), _i64(krows.size), _p(out))
    return out


def block_sums(A, B):
    """Exact integer sums of one contraction block, sum_j A[i, j] B[j, k], for
    code matrices A [m, <=128] and B [<=128, n] (|code| <= 127), through a
    library matmul in float32: every product is an integer of magnitude
    <= 127^2 and every partial sum of at most 128 of them stays below
    128 * 127^2 < 2^24, so it is an integer float32 holds exactly whatever
    the order of summation (and whatever the input rounding, since the codes
    are exact in any format with 7 significant bits).  A guard checks the row
    sums against integer arithmetic.  Returns a float64 torch tensor [m, n]."""
    import torch
    a = torch.from_numpy(np.ascontiguousarray(A, dtype=np.float32))
    b = torch.from_numpy(np.ascontiguousarray(B, dtype=np.float32))
    assert a.shape[1] == b.shape[0] <= TILE
    out = (a @ b).double()
    ref = np.asarray(A, dtype=np.int64) @ np.asarray(B, dtype=np.int64).sum(1)
    assert np.array_equal(out.sum(1).numpy(), ref.astype(np.float64)), "block sums are not exact"
    return out


def dx_matmul(Q, delta, W8, s_x, ec_mode, eps, rowsum, v, S, rows=None, tile=(TILE, TILE), chunk=2048):
    """The activation gradient of `dx` ([S3R] §III-A, §III-D) with each
    128-wide block's integer sum taken by `block_sums` (a library matmul)
    instead of nested loops.  The float64 promotion repeats `dx`'s order
    operation for operation -- blocks in ascending order, acc += delta *
    block, then eps * rowsum + v, then (acc - corr) / s_x, each a separately
    rounded IEEE operation -- so the result equals `dx` bit for bit; only the
    integer sums are formed differently."""
    import torch
    Q = np.asarray(Q, dtype=np.int8)
    W8 = np.asarray(W8, dtype=np.int8)
    T, N = Q.shape
    K = W8.shape[0]
    tr, tc = tile
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    nkb = -(-N // tc)
    delta = torch.from_numpy(np.asarray(delta, dtype=np.float32).astype(np.float64))
    out = np.zeros((rows.size, K), dtype=np.float64)
    Wt = [np.ascontiguousarray(W8[:, kb * tc:(kb + 1) * tc].T) for kb in range(nkb)]
    t64 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))
    for c0 in range(0, rows.size, chunk):
        r = rows[c0:c0 + chunk]
        tile_row = torch.from_numpy(r // tr)
        acc = torch.zeros((r.size, K), dtype=torch.float64)
        for kb in range(nkb):
            blk = block_sums(Q[r, kb * tc:(kb + 1) * tc], Wt[kb])
            acc += delta[tile_row, kb][:, None] * blk
        corr = torch.zeros_like(acc)
        if ec_mode in (EC_DX_ONLY, EC_TWO_WAY):
            corr = t64(eps)[r][:, None] * t64(rowsum)[None, :] + t64(v)[r // S]
        elif ec_mode == EC_DX_TOKEN_ONLY:
            corr = t64(eps)[r][:, None] * t64(rowsum)[None, :]
        sx = torch.ones(r.size, dtype=torch.float64) if s_x is None else \
            t64(np.asarray(s_x, dtype=np.float32)[r].astype(np.float64))
        out[c0:c0 + r.size] = ((acc - corr) / sx[:, None]).numpy()
    return out


def dw_matmul(X8, Q, delta, s_w, ec_mode, colmean, mu, xsum, p, S, krows=None, tile=(TILE, TILE)):
    """The weight gradient of `dw` ([S3R] §III-A, §III-D) with each 128-token
    block's integer sum taken by `block_sums`; the float64 promotion and the
    correction repeat `dw`'s order operation for operation (blocks in
    ascending order, then the per-example terms in example order, then p),
    so the result equals `dw` bit for bit."""
    import torch
    X8 = np.asarray(X8, dtype=np.int8)
    Q = np.asarray(Q, dtype=np.int8)
    T, K = X8.shape
    N = Q.shape[1]
    tr, tc = tile
    krows = np.arange(K) if krows is None else np.asarray(krows, dtype=np.int64)
    ntb = -(-T // tr)
    delta = np.asarray(delta, dtype=np.float32).astype(np.float64)
    acc = torch.zeros((krows.size, N), dtype=torch.float64)
    Xk = X8[:, krows]
    for tb in range(ntb):
        blk = block_sums(np.ascontiguousarray(Xk[tb * tr:(tb + 1) * tr].T), Q[tb * tr:(tb + 1) * tr])
        dcol = torch.from_numpy(np.repeat(delta[tb], tc)[:N])
        acc += dcol[None, :] * blk
    corr = torch.zeros_like(acc)
    t64 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))
    if ec_mode in (EC_TWO_WAY, EC_DW_ONLY):
        B = T // S
        xs, cm, m = t64(xsum), t64(colmean), t64(mu)
        kr = torch.from_numpy(krows)
        for b in range(B):
            corr += xs[b, kr][:, None] * (cm[b] - m[b])[None, :]
        corr += t64(p)[kr][:, None]
    sw = torch.ones(N, dtype=torch.float64) if s_w is None else \
        t64(np.asarray(s_w, dtype=np.float32).astype(np.float64))
    return ((acc - corr) / sw[None, :]).numpy()


def swiglu_bwd(dA, h1, h3):
    dA, h1, h3 = _f32(dA), _f32(h1), _f32(h3)
    dh1 = np.empty_like(dA)
    dh3 = np.empty_like(dA)
    lib().orc_swiglu_bwd(_p(dA), _p(h1), _p(h3), _i64(dA.size), _p(dh1), _p(dh3))
    return dh1, dh3


# --------------------------------------------------------------------------
# composition: one linear layer's backward ([S3R] §III-A .. §III-D)
# --------------------------------------------------------------------------
@dataclass
class LinearBackward:
    Q: np.ndarray              # codes used by dX (and dW unless independent SR)
    delta: np.ndarray
    E: np.ndarray
    Q_rhs: np.ndarray | None = None     # independent SR: codes used by dW
    delta_rhs: np.ndarray | None = None
    eps: np.ndarray | None = None
    colmean: np.ndarray | None = None
    mu: np.ndarray | None = None
    rowsum: np.ndarray | None = None
    v: np.ndarray | None = None
    xsum: np.ndarray | None = None
    p: np.ndarray | None = None
    dX: np.ndarray | None = None        # [len(rows), K] float64
    dW: np.ndarray | None = None        # [len(krows), N] float64
    status: int = 0
    extra: dict = field(default_factory=dict)


RHS_ID_OFFSET = 0x100   # tensor-id offset of the second (dW) copy under independent SR


def linear_backward(G, X8, s_x, W8, s_w, S, mode=S3R, ec_mode=EC_TWO_WAY, seed=0, tensor_id=0,
                    rows=None, krows=None, tile=(TILE, TILE), matmul=False) -> LinearBackward:
    """Backward of Y = X W given the saved forward operands.

    G: float32 [T, N] upstream gradient (exact widening of bf16).
    X8 [T, K] int8 with s_x [T]; W8 [K, N] int8 with s_w [N].
    rows / krows: which rows of dX / dW to produce (default: all).
    matmul: form the products' integer block sums with a library matmul
    (dx_matmul / dw_matmul, equal bit for bit) instead of nested loops.
    """
    G = _f32(G)
    T, N = G.shape
    K = W8.shape[0]
    rows = np.arange(T) if rows is None else np.asarray(rows)
    krows = np.arange(K) if krows is None else np.asarray(krows)
    Q, delta, E, st = quantize(G, s_x, s_w, mode, seed, tensor_id, tile, S=S)
    out = LinearBackward(Q=Q, delta=delta, E=E, status=st)
    use_ec = mode in SHARED and ec_mode != EC_NONE
    if mode == INDEP:
        Qr, dr, _, st2 = quantize(G, s_x, s_w, INDEP, seed, tensor_id + RHS_ID_OFFSET, tile)
        out.Q_rhs, out.delta_rhs, out.status = Qr, dr, st or st2
    if use_ec:
        out.eps, out.colmean, out.mu = error_stats(E, S)
        out.rowsum, out.v, out.xsum, out.p = ec_factors(out.eps, out.colmean, out.mu, S, W8,
                                                        X8 if ec_mode in (EC_TWO_WAY, EC_DW_ONLY) else None)
    em = ec_mode if use_ec else EC_NONE
    fdx, fdw = (dx_matmul, dw_matmul) if matmul else (dx, dw)
    out.dX = fdx(Q, delta, W8, s_x, em, out.eps, out.rowsum, out.v, S, rows, tile)
    Qw = out.Q_rhs if mode == INDEP else Q
    dw_delta = out.delta_rhs if mode == INDEP else delta
    out.dW = fdw(X8, Qw, dw_delta, s_w, em, out.colmean, out.mu, out.xsum, out.p, S, krows, tile)
    return out


# --------------------------------------------------------------------------
# composition: SwiGLU FFN block backward
# --------------------------------------------------------------------------
# Tensor ids of the three linears of one FFN block.
TID_W2, TID_W1, TID_W3 = 0, 1, 2


@dataclass
class FFNForwardOperands:
    X8: np.ndarray
    s_x: np.ndarray
    A8: np.ndarray
    s_a: np.ndarray
    W1_8: np.ndarray
    s_w1: np.ndarray
    W3_8: np.ndarray
    s_w3: np.ndarray
    W2_8: np.ndarray
    s_w2: np.ndarray


def gemm_fwd(X8, s_x, W8, s_w):
    """INT8 forward Y = diag(s_x) X8 W8 diag(s_w): the exact integer sum (S32
    accumulation), one rounding to fp32, then (acc * s_x) * s_w in fp32
    ([S3R] §III-A)."""
    X8 = np.ascontiguousarray(X8, dtype=np.int8)
    W8 = np.ascontiguousarray(W8, dtype=np.int8)
    T, K = X8.shape
    N = W8.shape[1]
    Y = np.zeros((T, N), dtype=np.float32)
    lib().orc_gemm_fwd(_p(X8), _p(_f32(s_x)), _p(W8), _p(_f32(s_w)), _i64(T), _i64(K), _i64(N), _p(Y))
    return Y


def to_bf16_bits(x) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even."""
    x = _f32(x)
    out = np.zeros(x.shape, dtype=np.uint16)
    for idx, v in np.ndenumerate(x):
        out[idx] = lib().orc_float_to_bf16(float(v))
    return out


def swiglu_fwd(h1f, h3f):
    """Forward gate: bf16 h1, h3 (bit patterns) and a = bf16(silu(h1) h3)."""
    h1f, h3f = _f32(h1f), _f32(h3f)
    h1b = np.zeros(h1f.shape, dtype=np.uint16)
    h3b = np.zeros(h1f.shape, dtype=np.uint16)
    ab = np.zeros(h1f.shape, dtype=np.uint16)
    lib().orc_swiglu_fwd(_p(h1f), _p(h3f), _i64(h1f.size), _p(h1b), _p(h3b), _p(ab))
    return h1b, h3b, ab


def sr_bf16_scalar(x: float, v: int) -> int:
    """bf16 bits of x rounded stochastically with the 16-bit threshold v."""
    return int(lib().orc_sr_bf16(float(x), int(v)))


def sr_bf16(X, mode=S3R, seed=0, tensor_id=0, t0=0) -> np.ndarray:
    """fp32 [T, N] -> bf16 bit patterns [T, N]: S3R (one 16-bit threshold per
    token), INDEP (one per element) or RTNE ([S3R] §II, §III-B).  Row i is
    token t0 + i."""
    X = _f32(X)
    T, N = X.shape
    Y = np.zeros((T, N), dtype=np.uint16)
    st = lib().orc_sr_bf16_matrix(_p(X), _i64(T), _i64(N), _i64(N), _i64(t0), C.c_int(mode), C.c_uint64(seed),
                                  C.c_uint32(tensor_id), _p(Y))
    if st != 0:
        raise ValueError(f"orc_sr_bf16_matrix status {st}")
    return Y


def sr_e4m3_scalar(y: float, v: int) -> int:
    """e4m3 code of y rounded stochastically with the 16-bit threshold v."""
    return int(lib().orc_sr_e4m3(float(y), int(v)))


def rn_e4m3_scalar(y: float) -> int:
    return int(lib().orc_rn_e4m3(float(y)))


def sr_fp8(X, inv_scale=1.0, mode=S3R, seed=0, tensor_id=0, t0=0) -> np.ndarray:
    """fp32 [T, N] -> e4m3 codes [T, N] of y = x * inv_scale (fp32): S3R (one
    16-bit threshold per token), INDEP (one per element) or RTNE ([S3R] §II,
    §III-B).  Row i is token t0 + i."""
    X = _f32(X)
    T, N = X.shape
    Y = np.zeros((T, N), dtype=np.uint8)
    st = lib().orc_sr_fp8_matrix(_p(X), _i64(T), _i64(N), _i64(N), _i64(t0), C.c_float(inv_scale), C.c_int(mode),
                                 C.c_uint64(seed), C.c_uint32(tensor_id), _p(Y))
    if st != 0:
        raise ValueError(f"orc_sr_fp8_matrix status {st}")
    return Y


@dataclass
class FFNForward:
    X8: np.ndarray
    s_x: np.ndarray
    W1_8: np.ndarray
    s_w1: np.ndarray
    W3_8: np.ndarray
    s_w3: np.ndarray
    W2_8: np.ndarray
    s_w2: np.ndarray
    h1: np.ndarray      # bf16 bit patterns [T, F]
    h3: np.ndarray
    a: np.ndarray
    A8: np.ndarray
    s_a: np.ndarray
    Y: np.ndarray       # fp32 [T, d]


def ffn_forward_int8(X, W1, W3, W2) -> FFNForward:
    """The SwiGLU block forward with INT8 GEMMs: RTNE operands (per-token X and
    a, per-output-channel weights), h1 = X W1 and h3 = X W3 saved as bf16,
    a = silu(h1) h3 in bf16, then Y = a W2 (fp32)."""
    X8, s_x = rtne_operand(X, 0)
    W1_8, s_w1 = rtne_operand(W1, 1)
    W3_8, s_w3 = rtne_operand(W3, 1)
    W2_8, s_w2 = rtne_operand(W2, 1)
    h1b, h3b, ab = swiglu_fwd(gemm_fwd(X8, s_x, W1_8, s_w1), gemm_fwd(X8, s_x, W3_8, s_w3))
    A8, s_a = rtne_operand(bf16_to_f32(ab), 0)
    Y = gemm_fwd(A8, s_a, W2_8, s_w2)
    return FFNForward(X8, s_x, W1_8, s_w1, W3_8, s_w3, W2_8, s_w2, h1b, h3b, ab, A8, s_a, Y)


def ffn_forward_operands(X, W1, W3, W2, a) -> FFNForwardOperands:
    """RTNE forward operands: per-token scales for X and a, per-output-channel
    scales for the weights ([S3R] §III-A)."""
    X8, s_x = rtne_operand(X, 0)
    A8, s_a = rtne_operand(a, 0)
    W1_8, s_w1 = rtne_operand(W1, 1)
    W3_8, s_w3 = rtne_operand(W3, 1)
    W2_8, s_w2 = rtne_operand(W2, 1)
    return FFNForwardOperands(X8, s_x, A8, s_a, W1_8, s_w1, W3_8, s_w3, W2_8, s_w2)


@dataclass
class FFNBackward:
    w2: LinearBackward
    w1: LinearBackward
    w3: LinearBackward
    dA: np.ndarray          # [T, F] float32 as fed to the glue (all rows)
    dh1: np.ndarray
    dh3: np.ndarray
    dX: np.ndarray          # [len(rows), d] float64
    dW1: np.ndarray
    dW2: np.ndarray
    dW3: np.ndarray


def ffn_backward(ops: FFNForwardOperands, h1, h3, dY, S, mode=S3R, ec_mode=EC_TWO_WAY, seed=0,
                 rows=None, krows_d=None, krows_f=None, tid_base=0, matmul=False) -> FFNBackward:
    """SwiGLU FFN block backward: W2 linear, then the SwiGLU glue, then W1 and
    W3 (dX = dX1 + dX3).  dA is needed for every token (the glue feeds the
    second quantization), so the W2 activation gradient is computed in full
    and rounded to fp32 before the glue, the precision the kernels hand on.
    The three linears use tensor ids tid_base + (0, 1, 2).  matmul: see
    linear_backward (the same results, fast enough for full-size blocks)."""
    T = dY.shape[0]
    F = ops.A8.shape[1]
    d = ops.X8.shape[1]
    rows = np.arange(T) if rows is None else np.asarray(rows)
    krows_d = np.arange(d) if krows_d is None else np.asarray(krows_d)
    krows_f = np.arange(F) if krows_f is None else np.asarray(krows_f)
    w2 = linear_backward(dY, ops.A8, ops.s_a, ops.W2_8, ops.s_w2, S, mode, ec_mode, seed, tid_base + TID_W2,
                         rows=np.arange(T), krows=krows_f, matmul=matmul)
    dA = w2.dX.astype(np.float32)
    dh1, dh3 = swiglu_bwd(dA, h1, h3)
    w1 = linear_backward(dh1, ops.X8, ops.s_x, ops.W1_8, ops.s_w1, S, mode, ec_mode, seed, tid_base + TID_W1,
                         rows=rows, krows=krows_d, matmul=matmul)
    w3 = linear_backward(dh3, ops.X8, ops.s_x, ops.W3_8, ops.s_w3, S, mode, ec_mode, seed, tid_base + TID_W3,
                         rows=rows, krows=krows_d, matmul=matmul)
    return FFNBackward(w2=w2, w1=w1, w3=w3, dA=dA, dh1=dh1, dh3=dh3,
                       dX=w1.dX + w3.dX, dW1=w1.dW, dW2=w2.dW, dW3=w3.dW)


# --------------------------------------------------------------------------
# grouped (mixture-of-experts) mode
# --------------------------------------------------------------------------
# Expert e's three linears use tensor ids MOE_TID_STRIDE * e + (W2, W1, W3).
MOE_TID_STRIDE = 16


@dataclass
class MoEForwardOperands:
    X8: np.ndarray      # [R, d] routed rows, expert-sorted, per-row scales
    s_x: np.ndarray
    A8: np.ndarray      # [R, F]
    s_a: np.ndarray
    W1_8: np.ndarray    # [E, d, F], per-expert per-output-channel scales [E, F]
    s_w1: np.ndarray
    W3_8: np.ndarray
    s_w3: np.ndarray
    W2_8: np.ndarray    # [E, F, d], scales [E, d]
    s_w2: np.ndarray

    def expert(self, e: int, r0: int, r1: int) -> FFNForwardOperands:
        return FFNForwardOperands(self.X8[r0:r1], self.s_x[r0:r1], self.A8[r0:r1], self.s_a[r0:r1],
                                  self.W1_8[e], self.s_w1[e], self.W3_8[e], self.s_w3[e], self.W2_8[e],
                                  self.s_w2[e])


def moe_forward_operands(X, W1, W3, W2, a) -> MoEForwardOperands:
    """RTNE forward operands of the routed rows (per-row scales) and of every
    expert's weights (per-output-channel scales within the expert)."""
    X8, s_x = rtne_operand(X, 0)
    A8, s_a = rtne_operand(a, 0)
    w = [[rtne_operand(Wk[e], 1) for e in range(Wk.shape[0])] for Wk in (W1, W3, W2)]
    st = lambda k, i: np.stack([w[k][e][i] for e in range(len(w[k]))])
    return MoEForwardOperands(X8, s_x, A8, s_a, st(0, 0), st(0, 1), st(1, 0), st(1, 1), st(2, 0), st(2, 1))


@dataclass
class MoEBackward:
    dX: np.ndarray      # [R, d] float64 (zero-size groups leave no rows)
    dW1: np.ndarray     # [E, d, F] float64 (an empty expert's gradients are zero)
    dW3: np.ndarray
    dW2: np.ndarray     # [E, F, d]
    experts: list       # FFNBackward per expert (None for an empty group)


def moe_ffn_backward(ops: MoEForwardOperands, h1, h3, dY, offsets, mode=S3R, ec_mode=EC_TWO_WAY,
                     seed=0, matmul=False) -> MoEBackward:
    """Grouped SwiGLU FFN backward over expert-sorted routed rows ([S3R] §IV,
    MoE models): expert e owns rows offsets[e] .. offsets[e+1] and runs the
    whole block backward on them as one example, with its own weights; tiles
    and token indices restart at the group's first row, and its tensor ids
    are MOE_TID_STRIDE * e + (0, 1, 2)."""
    E = ops.W1_8.shape[0]
    R, d = ops.X8.shape
    F = ops.A8.shape[1]
    dX = np.zeros((R, d))
    dW1, dW3, dW2 = np.zeros((E, d, F)), np.zeros((E, d, F)), np.zeros((E, F, d))
    per = []
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            per.append(None)
            continue
        b = ffn_backward(ops.expert(e, r0, r1), h1[r0:r1], h3[r0:r1], dY[r0:r1], r1 - r0, mode, ec_mode, seed,
                         tid_base=MOE_TID_STRIDE * e, matmul=matmul)
        dX[r0:r1] = b.dX
        dW1[e], dW3[e], dW2[e] = b.dW1, b.dW3, b.dW2
        per.append(b)
    return MoEBackward(dX, dW1, dW3, dW2, per)
