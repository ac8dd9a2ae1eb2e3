"""Python binding of libs3r: the S3R / S3R-EC INT8 backward on GB300 (sm_103a).

Argument marshalling only: every step of the backward runs in the CUDA kernels
of ``libs3r.so`` (built in-tree by ``build.py``).  PyTorch supplies device
memory and the current stream.  There is no CPU fallback: if the library is
missing or no GPU is present, calls raise.

The functions carry the C ABI's names (see ``include/s3r.h`` for the exact
semantics, layouts and citations):

    s3r_quantize, indep_sr_quantize, rtne_quantize, swiglu_quantize,
    s3r_ec_correct, int8_gemm_dx, int8_gemm_dx_sum, int8_gemm_dw, ffn_backward

Outputs may be passed in (then they are written in place) or are allocated
with torch on the inputs' device.  Codes are int8 tensors (S3R_CODES_S8) or
float16 tensors holding the same integers (S3R_CODES_F16, the operand format
of the tcgen05 GEMMs); the format follows the tensors' dtype.
"""
from __future__ import annotations

import ctypes as C
import os
import re
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libs3r.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "s3r.h")
TILE = 128

S3R_OK = 0
ROUND_RTNE, ROUND_S3R, ROUND_INDEP, ROUND_S3R_7BIT, ROUND_BCAST = 0, 1, 2, 3, 4
EC_NONE, EC_DX_ONLY, EC_TWO_WAY, EC_DW_ONLY = 0, 1, 2, 3
AXIS_ROW, AXIS_COL, AXIS_TILE = 0, 1, 2
TID_W2, TID_W1, TID_W3, RHS_ID_OFFSET = 0, 1, 2, 0x100
MOE_TID_STRIDE = 16   # grouped mode: expert e uses tensor ids 16 e + (0, 1, 2)
CODES_S8, CODES_F16 = 0, 1
CODES_S8_F16 = 2   # ffn_backward only: int8 operand codes widened to fp16 inside the call
DEFAULT_CODES = CODES_F16
_CODE_DTYPE = {CODES_S8: torch.int8, CODES_F16: torch.float16, CODES_S8_F16: torch.float16}

_lib = None

_VP, _I64, _U64, _U32, _INT, _SZ = C.c_void_p, C.c_int64, C.c_uint64, C.c_uint32, C.c_int, C.c_size_t

_SIGS = {
    "s3r_status_string": (C.c_char_p, [_INT]),
    "s3r_abi_version": (_INT, []),
    "s3r_kernel_launch_count": (C.c_uint64, []),
    "s3r_last_error": (C.c_char_p, []),
    "s3r_quantize": (_INT, [_VP, _I64, _I64, _I64, _VP, _VP, _U64, _U32, _VP, _INT, _VP, _VP, _VP, _VP, _VP]),
    "s3r_quantize_ex": (_INT, [_VP, _I64, _I64, _I64, _VP, _VP, _INT, _I64, _VP, _U64, _U32, _VP, _INT, _VP, _VP,
                               _VP, _VP, _VP]),
    "indep_sr_quantize": (_INT, [_VP, _I64, _I64, _I64, _VP, _VP, _U64, _U32, _VP, _INT, _VP, _VP, _VP]),
    "rtne_quantize": (_INT, [_VP, _I64, _I64, _I64, _VP, _VP, _INT, _VP, _INT, _VP, _VP, _VP]),
    "swiglu_quantize": (_INT, [_VP, _I64, _VP, _VP, _I64, _I64, _I64, _VP, _VP, _VP, _INT, _INT, _U64, _U32, _U32,
                               _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "swiglu_quantize_ex": (_INT, [_VP, _I64, _VP, _VP, _I64, _I64, _I64, _VP, _VP, _VP, _INT, _I64, _INT, _U64, _U32,
                                  _U32, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "s3r_ec_workspace_size": (_SZ, [_I64, _I64]),
    "s3r_ec_correct": (_INT, [_VP, _VP, _I64, _I64, _I64, _VP, _I64, _VP, _INT, _INT, _VP, _VP, _VP, _VP, _VP, _VP,
                              _VP, _VP, _SZ, _VP, _VP]),
    "s3r_ec_correct_static": (_INT, [_VP, _VP, _I64, _I64, _I64, _VP, _I64, _VP, _INT, _INT, _VP, _VP, _VP, _VP, _VP,
                                     _VP, _VP, _VP, _VP]),
    "int8_gemm_dx": (_INT, [_VP, _VP, _VP, _INT, _I64, _I64, _I64, _VP, _INT, _VP, _VP, _VP, _I64, _VP, _INT, _VP,
                            _VP]),
    "int8_gemm_dx_sum": (_INT, [_VP, _INT, _INT, _I64, _I64, _I64, _VP, _INT, _I64, _VP, _INT, _VP, _VP]),
    "int8_gemm_dw_workspace_size": (_SZ, [_I64, _I64, _I64, _INT]),
    "int8_gemm_dw": (_INT, [_VP, _VP, _VP, _INT, _I64, _I64, _I64, _VP, _INT, _VP, _VP, _VP, _VP, _I64, _VP, _VP,
                            _SZ, _VP, _VP]),
    "int8_gemm_fwd": (_INT, [_VP, _VP, _VP, _VP, _INT, _I64, _I64, _I64, _VP, _VP, _VP]),
    "int8_gemm_fwd_swiglu": (_INT, [_VP, _VP, _VP, _VP, _VP, _VP, _INT, _I64, _I64, _I64, _VP, _VP, _VP, _VP,
                                    _VP]),
    "swiglu_fwd_quantize": (_INT, [_VP, _VP, _I64, _I64, _I64, _VP, _VP, _INT, _VP, _VP, _VP]),
    "ffn_forward": (_INT, [_VP, _VP]),
    "s3r_sr_bf16": (_INT, [_VP, _I64, _I64, _I64, _INT, _U64, _U32, _VP, _I64, _VP]),
    "s3r_sr_fp8": (_INT, [_VP, _I64, _I64, _I64, C.c_float, _INT, _U64, _U32, _VP, _I64, _VP]),
    "s3r_ffn_workspace_size": (_SZ, [_I64, _I64, _I64, _I64, _INT, _INT, _INT]),
    "s3r_ffn_grouped_workspace_size": (_SZ, [_VP, _I64, _I64, _I64, _INT, _INT, _INT]),
    "s3r_ffn_workspace_size_flags": (_SZ, [_I64, _I64, _I64, _I64, _INT, _INT, _INT, _INT]),
    "s3r_ffn_grouped_workspace_size_flags": (_SZ, [_VP, _I64, _I64, _I64, _INT, _INT, _INT, _INT]),
    "ffn_backward": (_INT, [_VP, _VP]),
    "s3r_ffn_workspace_offsets": (_INT, [_I64, _I64, _I64, _I64, _INT, _INT, _VP, _I64, _I64, _VP]),
    "s3r_debug_dx_blocks": (_INT, [_VP, _VP, _INT, _I64, _I64, _I64, _VP, _VP]),
    "s3r_check_reciprocal": (_INT, [_U32, _U32, _VP, _VP]),
    "s3r_debug_wait_timeout": (_INT, [_INT, _U64, _INT, _VP, _VP, _VP]),
    "s3r_debug_dw_blocks": (_INT, [_VP, _VP, _INT, _I64, _I64, _I64, _VP, _VP, _SZ, _VP]),
}


class S3RError(RuntimeError):
    pass


def header_functions() -> list[str]:
    """Names of every function the C header declares."""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?(?:int|size_t|uint64_t|char\s*\*|const\s+char\s*\*)\s*\**\s*(\w+)\s*\(",
                      txt, re.M)


def kernel_launch_count() -> int:
    """Kernels launched by libs3r so far in this process."""
    return int(lib().s3r_kernel_launch_count())


def lib():
    """Load libs3r.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise S3RError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().s3r_status_string(int(code)).decode()


def _check(code: int, what: str):
    if code != S3R_OK:
        detail = lib().s3r_last_error().decode()
        raise S3RError(f"{what}: {status_string(code)}" + (f" [{detail}]" if detail else ""))


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise S3RError("libs3r takes device tensors only")
    return C.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _cdiv(a, b):
    return -(-a // b)


def new_status(device="cuda") -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def check_status(status: torch.Tensor):
    """Synchronize-free read is not possible: this copies the device status to the host."""
    code = int(status.item())
    _check(code, "device status")


def _bits(t):
    assert t.dtype == torch.bfloat16, t.dtype
    return t


def code_format_of(t) -> int:
    """S3R_CODES_* of a code tensor, from its dtype."""
    if t.dtype == torch.int8:
        return CODES_S8
    if t.dtype == torch.float16:
        return CODES_F16
    raise S3RError(f"codes must be int8 or float16, got {t.dtype}")


def _fmt2(a, b) -> int:
    fa, fb = code_format_of(a), code_format_of(b)
    if fa != fb:
        raise S3RError("both operands of a product must use the same code format")
    return fa


# ---------------------------------------------------------------------------
# quantizers
# ---------------------------------------------------------------------------
@dataclass
class Quantized:
    Q: torch.Tensor
    tile_scale: torch.Tensor
    tok_err_part: torch.Tensor | None = None
    col_err_part: torch.Tensor | None = None


def s3r_quantize(G, s_x=None, s_w=None, seed=0, tensor_id=0, out: Quantized | None = None, partials=True,
                 status=None, stream=None, code_format=DEFAULT_CODES) -> Quantized:
    T, N = G.shape
    dev = G.device
    if out is None:
        out = Quantized(torch.empty((T, N), dtype=_CODE_DTYPE[code_format], device=dev),
                        torch.empty((_cdiv(T, TILE), _cdiv(N, TILE)), dtype=torch.float32, device=dev),
                        torch.empty((T, _cdiv(N, TILE)), dtype=torch.float32, device=dev) if partials else None,
                        torch.empty((_cdiv(T, TILE), N), dtype=torch.float32, device=dev) if partials else None)
    _check(lib().s3r_quantize(_ptr(_bits(G)), T, N, G.stride(0), _ptr(s_x), _ptr(s_w), seed, tensor_id, _ptr(out.Q),
                              code_format_of(out.Q), _ptr(out.tile_scale), _ptr(out.tok_err_part),
                              _ptr(out.col_err_part), _ptr(status), _stream(stream)), "s3r_quantize")
    return out


def s3r_quantize_ex(G, s_x=None, s_w=None, round_mode=ROUND_S3R, S=0, per_tensor=False, seed=0, tensor_id=0,
                    out: Quantized | None = None, partials=True, status=None, stream=None,
                    code_format=DEFAULT_CODES):
    """s3r_quantize with a rounding mode, S tokens per example (Phi_bcast) and an
    optional per-tensor step; returns (Quantized, tensor_amax or None)."""
    T, N = G.shape
    dev = G.device
    if out is None:
        out = Quantized(torch.empty((T, N), dtype=_CODE_DTYPE[code_format], device=dev),
                        torch.empty((_cdiv(T, TILE), _cdiv(N, TILE)), dtype=torch.float32, device=dev),
                        torch.empty((T, _cdiv(N, TILE)), dtype=torch.float32, device=dev) if partials else None,
                        torch.empty((_cdiv(T, TILE), N), dtype=torch.float32, device=dev) if partials else None)
    amax = torch.empty(1, dtype=torch.float32, device=dev) if per_tensor else None
    _check(lib().s3r_quantize_ex(_ptr(_bits(G)), T, N, G.stride(0), _ptr(s_x), _ptr(s_w), round_mode, S, _ptr(amax),
                                 seed, tensor_id, _ptr(out.Q), code_format_of(out.Q), _ptr(out.tile_scale),
                                 _ptr(out.tok_err_part), _ptr(out.col_err_part), _ptr(status), _stream(stream)),
           "s3r_quantize_ex")
    return out, amax


def indep_sr_quantize(G, s_x=None, s_w=None, seed=0, tensor_id=0, out: Quantized | None = None, status=None,
                      stream=None, code_format=DEFAULT_CODES) -> Quantized:
    T, N = G.shape
    dev = G.device
    if out is None:
        out = Quantized(torch.empty((T, N), dtype=_CODE_DTYPE[code_format], device=dev),
                        torch.empty((_cdiv(T, TILE), _cdiv(N, TILE)), dtype=torch.float32, device=dev))
    _check(lib().indep_sr_quantize(_ptr(_bits(G)), T, N, G.stride(0), _ptr(s_x), _ptr(s_w), seed, tensor_id,
                                   _ptr(out.Q), code_format_of(out.Q), _ptr(out.tile_scale), _ptr(status),
                                   _stream(stream)),
           "indep_sr_quantize")
    return out


def rtne_quantize(A, scale_axis=AXIS_TILE, s_x=None, s_w=None, Q=None, scale=None, status=None, stream=None,
                  code_format=DEFAULT_CODES):
    R, Cc = A.shape
    dev = A.device
    if Q is None:
        Q = torch.empty((R, Cc), dtype=_CODE_DTYPE[code_format], device=dev)
    if scale is None:
        shape = {AXIS_ROW: (R,), AXIS_COL: (Cc,), AXIS_TILE: (_cdiv(R, TILE), _cdiv(Cc, TILE))}[scale_axis]
        scale = torch.empty(shape, dtype=torch.float32, device=dev)
    _check(lib().rtne_quantize(_ptr(_bits(A)), R, Cc, A.stride(0), _ptr(s_x), _ptr(s_w), scale_axis, _ptr(Q),
                               code_format_of(Q), _ptr(scale), _ptr(status), _stream(stream)), "rtne_quantize")
    return Q, scale


def swiglu_quantize(dA, h1, h3, s_x=None, s_w1=None, s_w3=None, round_mode=ROUND_S3R, seed=0, tid1=TID_W1,
                    tid3=TID_W3, partials=True, status=None, stream=None, code_format=DEFAULT_CODES, S=0):
    T, F = dA.shape
    dev = dA.device

    def mk():
        return Quantized(torch.empty((T, F), dtype=_CODE_DTYPE[code_format], device=dev),
                         torch.empty((_cdiv(T, TILE), _cdiv(F, TILE)), dtype=torch.float32, device=dev),
                         torch.empty((T, _cdiv(F, TILE)), dtype=torch.float32, device=dev) if partials else None,
                         torch.empty((_cdiv(T, TILE), F), dtype=torch.float32, device=dev) if partials else None)

    o1, o3 = mk(), mk()
    assert dA.dtype == torch.float32 and h1.stride(0) == h3.stride(0)
    _check(lib().swiglu_quantize_ex(_ptr(dA), dA.stride(0), _ptr(_bits(h1)), _ptr(_bits(h3)), h1.stride(0), T, F,
                                    _ptr(s_x), _ptr(s_w1), _ptr(s_w3), round_mode, S, code_format, seed, tid1, tid3,
                                    _ptr(o1.Q), _ptr(o1.tile_scale), _ptr(o1.tok_err_part), _ptr(o1.col_err_part),
                                    _ptr(o3.Q), _ptr(o3.tile_scale), _ptr(o3.tok_err_part), _ptr(o3.col_err_part),
                                    _ptr(status), _stream(stream)), "swiglu_quantize")
    return o1, o3


# ---------------------------------------------------------------------------
# error correction
# ---------------------------------------------------------------------------
@dataclass
class ECFactors:
    eps: torch.Tensor
    mu: torch.Tensor
    colmean: torch.Tensor
    rowsum: torch.Tensor | None
    v: torch.Tensor | None
    xsum: torch.Tensor | None
    p: torch.Tensor | None


def s3r_ec_correct(q: Quantized, T, N, S, W8=None, X8=None, ec_mode=EC_TWO_WAY, status=None, stream=None) -> ECFactors:
    dev = q.Q.device
    B = T // S
    K = W8.shape[0] if W8 is not None else 0
    f = lambda *s: torch.empty(s, dtype=torch.float32, device=dev)
    i = lambda *s: torch.empty(s, dtype=torch.int32, device=dev)
    ec = ECFactors(f(T), f(B), f(B, N), i(K) if K else None, f(B, K) if K else None,
                   i(B, K) if ec_mode in (EC_TWO_WAY, EC_DW_ONLY) else None,
                   f(K) if ec_mode in (EC_TWO_WAY, EC_DW_ONLY) else None)
    ws_bytes = lib().s3r_ec_workspace_size(T, K) if ec_mode in (EC_TWO_WAY, EC_DW_ONLY) else 0
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    fmt = code_format_of(W8 if W8 is not None else q.Q)
    _check(lib().s3r_ec_correct(_ptr(q.tok_err_part), _ptr(q.col_err_part), T, N, S, _ptr(W8), K, _ptr(X8), fmt, ec_mode,
                                _ptr(ec.eps), _ptr(ec.mu), _ptr(ec.colmean), _ptr(ec.rowsum), _ptr(ec.v),
                                _ptr(ec.xsum), _ptr(ec.p), _ptr(ws), ws_bytes, _ptr(status), _stream(stream)),
           "s3r_ec_correct")
    return ec


# ---------------------------------------------------------------------------
# GEMMs
# ---------------------------------------------------------------------------
def int8_gemm_dx(Q, tile_scale, W8, s_x=None, ec_mode=EC_NONE, ec: ECFactors | None = None, S=None, dX=None,
                 accumulate=False, status=None, stream=None):
    T, N = Q.shape
    K = W8.shape[0]
    if dX is None:
        dX = torch.empty((T, K), dtype=torch.float32, device=Q.device)
    S = T if S is None else S
    _check(lib().int8_gemm_dx(_ptr(Q), _ptr(tile_scale), _ptr(W8), _fmt2(Q, W8), T, N, K, _ptr(s_x), ec_mode,
                              _ptr(ec.eps if ec else None), _ptr(ec.rowsum if ec else None),
                              _ptr(ec.v if ec else None), S, _ptr(dX), int(accumulate), _ptr(status),
                              _stream(stream)), "int8_gemm_dx")
    return dX


class _DxTerm(C.Structure):
    """struct s3r_dx_term"""
    _fields_ = [("Q", _VP), ("tile_scale", _VP), ("W8", _VP), ("eps", _VP), ("rowsum", _VP), ("v", _VP)]


DX_MAX_TERMS = 2


def int8_gemm_dx_sum(terms, s_x=None, ec_mode=EC_NONE, S=None, dX=None, accumulate=False, status=None,
                     stream=None):
    """dX = sum over terms of the corrected, rescaled Q_i W8_i^T; `terms` is a
    list of (Q, tile_scale, W8, ec) with ec an ECFactors or None."""
    if not 1 <= len(terms) <= DX_MAX_TERMS:
        raise S3RError(f"int8_gemm_dx_sum takes 1..{DX_MAX_TERMS} terms")
    Q0, _, W0, _ = terms[0]
    T, N = Q0.shape
    K = W0.shape[0]
    for Q, _, W8, _ in terms:
        if tuple(Q.shape) != (T, N) or tuple(W8.shape) != (K, N):
            raise S3RError("int8_gemm_dx_sum: every term needs Q [T, N] and W8 [K, N] of the same sizes")
    fmt = _fmt2(Q0, W0)
    if dX is None:
        dX = torch.empty((T, K), dtype=torch.float32, device=Q0.device)
    S = T if S is None else S
    arr = (_DxTerm * len(terms))()
    for i, (Q, sc, W8, ec) in enumerate(terms):
        if _fmt2(Q, W8) != fmt:
            raise S3RError("int8_gemm_dx_sum: every term needs the same code format")
        arr[i] = _DxTerm(_ptr(Q), _ptr(sc), _ptr(W8), _ptr(ec.eps if ec else None),
                         _ptr(ec.rowsum if ec else None), _ptr(ec.v if ec else None))
    _check(lib().int8_gemm_dx_sum(C.cast(arr, _VP), len(terms), fmt, T, N, K, _ptr(s_x), ec_mode, S, _ptr(dX),
                                  int(accumulate), _ptr(status), _stream(stream)), "int8_gemm_dx_sum")
    return dX


def int8_gemm_dw(X8, Q, tile_scale, s_w=None, ec_mode=EC_NONE, ec: ECFactors | None = None, S=None, dW=None,
                 workspace=None, status=None, stream=None):
    T, K = X8.shape
    N = Q.shape[1]
    if dW is None:
        dW = torch.empty((K, N), dtype=torch.float32, device=Q.device)
    fmt = _fmt2(X8, Q)
    ws_bytes = lib().int8_gemm_dw_workspace_size(T, K, N, fmt)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=Q.device)
    S = T if S is None else S
    two = ec_mode in (EC_TWO_WAY, EC_DW_ONLY) and ec is not None
    _check(lib().int8_gemm_dw(_ptr(X8), _ptr(Q), _ptr(tile_scale), fmt, T, K, N, _ptr(s_w), ec_mode,
                              _ptr(ec.colmean if two else None), _ptr(ec.mu if two else None),
                              _ptr(ec.xsum if two else None), _ptr(ec.p if two else None), S, _ptr(dW),
                              _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream)), "int8_gemm_dw")
    return dW


def check_reciprocal(lo_bits, hi_bits, device="cuda", stream=None) -> int:
    """Floats with bit patterns in [lo_bits, hi_bits) whose reciprocal in the
    SwiGLU glue differs from the IEEE one (test hook)."""
    count = torch.zeros(1, dtype=torch.int64, device=device)
    _check(lib().s3r_check_reciprocal(lo_bits, hi_bits, _ptr(count), _stream(stream)), "s3r_check_reciprocal")
    return int(count.item())


WAIT_GEMM, WAIT_QUANTIZE, WAIT_EC = 0, 1, 2


def debug_wait_timeout(family, limit_ns, raise_abort=False, device="cuda", stream=None):
    """Run one kernel family's bounded wait on a barrier that nothing arrives
    on (test hook): returns (device status, nanoseconds waited)."""
    st = torch.zeros(1, dtype=torch.int32, device=device)
    waited = torch.zeros(1, dtype=torch.int64, device=device)
    _check(lib().s3r_debug_wait_timeout(family, limit_ns, int(bool(raise_abort)), _ptr(st), _ptr(waited),
                                        _stream(stream)), "s3r_debug_wait_timeout")
    torch.cuda.synchronize()
    return int(st.item()), int(waited.item())


def debug_dx_blocks(Q, W8, stream=None):
    T, N = Q.shape
    K = W8.shape[0]
    out = torch.empty((T, K, _cdiv(N, TILE)), dtype=torch.int32, device=Q.device)
    _check(lib().s3r_debug_dx_blocks(_ptr(Q), _ptr(W8), _fmt2(Q, W8), T, N, K, _ptr(out), _stream(stream)),
           "s3r_debug_dx_blocks")
    return out


def debug_dw_blocks(X8, Q, stream=None):
    T, K = X8.shape
    N = Q.shape[1]
    out = torch.empty((K, N, _cdiv(T, TILE)), dtype=torch.int32, device=Q.device)
    fmt = _fmt2(X8, Q)
    ws_bytes = lib().int8_gemm_dw_workspace_size(T, K, N, fmt)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=Q.device)
    _check(lib().s3r_debug_dw_blocks(_ptr(X8), _ptr(Q), fmt, T, K, N, _ptr(out), _ptr(ws), ws.numel(),
                                     _stream(stream)), "s3r_debug_dw_blocks")
    return out


# ---------------------------------------------------------------------------
# forward GEMMs
# ---------------------------------------------------------------------------
def int8_gemm_fwd(X8, s_x, W8, s_w, Y=None, status=None, stream=None):
    """Y = (X8 W8 * s_x[t]) * s_w[n] in fp32; X8 [T, K], W8 [K, N] fp16 codes."""
    T, K = X8.shape
    N = W8.shape[1]
    if Y is None:
        Y = torch.empty((T, N), dtype=torch.float32, device=X8.device)
    _check(lib().int8_gemm_fwd(_ptr(X8), _ptr(s_x), _ptr(W8), _ptr(s_w), _fmt2(X8, W8), T, K, N, _ptr(Y),
                               _ptr(status), _stream(stream)), "int8_gemm_fwd")
    return Y


def int8_gemm_fwd_swiglu(X8, s_x, W1_8, s_w1, W3_8, s_w3, h1=None, h3=None, a=None, with_gate=True, status=None,
                         stream=None):
    """The gate and up projections (and, with_gate, the SwiGLU gate in the
    epilogue): returns bf16 (h1, h3, a or None)."""
    T, K = X8.shape
    F = W1_8.shape[1]
    new = lambda: torch.empty((T, F), dtype=torch.bfloat16, device=X8.device)
    out = [h1 if h1 is not None else new(), h3 if h3 is not None else new(),
           (a if a is not None else new()) if with_gate else None]
    _check(lib().int8_gemm_fwd_swiglu(_ptr(X8), _ptr(s_x), _ptr(W1_8), _ptr(s_w1), _ptr(W3_8), _ptr(s_w3),
                                      _fmt2(X8, W1_8), T, K, F, _ptr(out[0]), _ptr(out[1]), _ptr(out[2]),
                                      _ptr(status), _stream(stream)), "int8_gemm_fwd_swiglu")
    return tuple(out)


def swiglu_fwd_quantize(h1, h3, a=None, keep_a=True, Q=None, scale=None, status=None, stream=None,
                        code_format=DEFAULT_CODES):
    """a = bf16(silu(h1) h3) fused into its per-token RTNE: returns (a or None, Q, scale)."""
    T, F = h1.shape
    assert h1.shape == h3.shape and h1.stride(0) == h3.stride(0)
    dev = h1.device
    if keep_a and a is None:
        a = torch.empty((T, F), dtype=torch.bfloat16, device=dev)
    if Q is None:
        Q = torch.empty((T, F), dtype=_CODE_DTYPE[code_format], device=dev)
    if scale is None:
        scale = torch.empty((T,), dtype=torch.float32, device=dev)
    _check(lib().swiglu_fwd_quantize(_ptr(_bits(h1)), _ptr(_bits(h3)), T, F, h1.stride(0),
                                     _ptr(a if keep_a else None), _ptr(Q), code_format_of(Q), _ptr(scale),
                                     _ptr(status), _stream(stream)), "swiglu_fwd_quantize")
    return (a if keep_a else None), Q, scale


def s3r_sr_bf16(X, round_mode=ROUND_S3R, seed=0, tensor_id=0, Y=None, stream=None):
    """fp32 [T, N] -> bf16 [T, N], stochastically rounded with one 16-bit
    threshold per token (ROUND_S3R), per element (ROUND_INDEP), or RTNE."""
    assert X.dtype == torch.float32 and X.dim() == 2
    T, N = X.shape
    if Y is None:
        Y = torch.empty((T, N), dtype=torch.bfloat16, device=X.device)
    _check(lib().s3r_sr_bf16(_ptr(X), T, N, X.stride(0), round_mode, seed, tensor_id, _ptr(Y), Y.stride(0),
                             _stream(stream)), "s3r_sr_bf16")
    return Y


def s3r_sr_fp8(X, inv_scale=1.0, round_mode=ROUND_S3R, seed=0, tensor_id=0, Y=None, stream=None):
    """fp32 [T, N] -> e4m3 codes [T, N] (uint8) of X * inv_scale, stochastically
    rounded with one 16-bit threshold per token (ROUND_S3R), per element
    (ROUND_INDEP), or RTNE; saturating at +-448."""
    assert X.dtype == torch.float32 and X.dim() == 2
    T, N = X.shape
    if Y is None:
        Y = torch.empty((T, N), dtype=torch.uint8, device=X.device)
    _check(lib().s3r_sr_fp8(_ptr(X), T, N, X.stride(0), float(inv_scale), round_mode, seed, tensor_id, _ptr(Y),
                            Y.stride(0), _stream(stream)), "s3r_sr_fp8")
    return Y


class _FfnFwdArgs(C.Structure):
    _fields_ = [("T", C.c_int64), ("d", C.c_int64), ("F", C.c_int64),
                ("X", _VP), ("W1", _VP), ("W3", _VP), ("W2", _VP),
                ("quantize_weights", C.c_int), ("code_format", C.c_int),
                ("X8", _VP), ("s_x", _VP), ("W1_8", _VP), ("s_w1", _VP), ("W3_8", _VP), ("s_w3", _VP),
                ("W2_8", _VP), ("s_w2", _VP), ("h1", _VP), ("h3", _VP), ("a", _VP), ("A8", _VP), ("s_a", _VP),
                ("Y", _VP), ("d_status", _VP)]


@dataclass
class FFNForward:
    """The block forward's outputs: the backward's operands, a (or None: the
    backward reads only its codes) and Y."""
    ops: "FFNOperands"
    a: torch.Tensor | None
    Y: torch.Tensor


def alloc_ffn_forward(T, d, F, device="cuda", keep_a=True) -> FFNForward:
    """Output buffers of ffn_forward (fp16 codes)."""
    e = lambda *shape, dt=torch.float16: torch.empty(shape, dtype=dt, device=device)
    f32, bf = torch.float32, torch.bfloat16
    ops = FFNOperands(e(T, d), e(T, dt=f32), e(T, F), e(T, dt=f32), e(d, F), e(F, dt=f32), e(d, F), e(F, dt=f32),
                      e(F, d), e(d, dt=f32), e(T, F, dt=bf), e(T, F, dt=bf))
    return FFNForward(ops, e(T, F, dt=bf) if keep_a else None, e(T, d, dt=f32))


def ffn_forward(X, W1=None, W3=None, W2=None, out: FFNForward | None = None, quantize_weights=True, status=None,
                stream=None, keep_a=True) -> FFNForward:
    """The SwiGLU block forward with INT8 GEMMs (one C call, five launches):
    RTNE X and (unless quantize_weights is False, in which case `out.ops`
    already holds the weights' codes) the weights, h1/h3/a through the fused
    gate, RTNE a, Y = a W2."""
    T, d = X.shape
    F = out.ops.W1_8.shape[1] if out is not None else W1.shape[1]
    if out is None:
        out = alloc_ffn_forward(T, d, F, X.device, keep_a)
    o = out.ops
    args = _FfnFwdArgs(T, d, F, _ptr(_bits(X)), _ptr(_bits(W1) if W1 is not None else None),
                       _ptr(_bits(W3) if W3 is not None else None), _ptr(_bits(W2) if W2 is not None else None),
                       int(quantize_weights), CODES_F16, _ptr(o.X8), _ptr(o.s_x), _ptr(o.W1_8), _ptr(o.s_w1),
                       _ptr(o.W3_8), _ptr(o.s_w3), _ptr(o.W2_8), _ptr(o.s_w2), _ptr(o.h1), _ptr(o.h3), _ptr(out.a),
                       _ptr(o.A8), _ptr(o.s_a), _ptr(out.Y), _ptr(status))
    _check(lib().ffn_forward(C.byref(args), _stream(stream)), "ffn_forward")
    return out


# ---------------------------------------------------------------------------
# whole FFN block
# ---------------------------------------------------------------------------
class _FfnArgs(C.Structure):
    _fields_ = [("T", C.c_int64), ("d", C.c_int64), ("F", C.c_int64), ("S", C.c_int64),
                ("dY", _VP), ("h1", _VP), ("h3", _VP),
                ("X8", _VP), ("s_x", _VP), ("A8", _VP), ("s_a", _VP),
                ("W1_8", _VP), ("s_w1", _VP), ("W3_8", _VP), ("s_w3", _VP), ("W2_8", _VP), ("s_w2", _VP),
                ("round_mode", C.c_int), ("ec_mode", C.c_int), ("code_format", C.c_int), ("seed", C.c_uint64),
                ("dX", _VP), ("dW1", _VP), ("dW3", _VP), ("dW2", _VP),
                ("workspace", _VP), ("workspace_bytes", C.c_size_t), ("d_status", _VP),
                ("step_events", C.POINTER(C.c_void_p)), ("num_groups", C.c_int64),
                ("group_offsets", C.POINTER(C.c_int64)), ("flags", C.c_int)]


FFN_NUM_EVENTS = 9
FFN_FUSE_GLUE = 1   # S3R_FFN_FUSE_GLUE
FFN_RECOMPUTE_A = 2   # S3R_FFN_RECOMPUTE_A
FFN_STEPS = ["quantize dY", "EC W2", "GEMM dA (dX of W2)", "GEMM dW2", "SwiGLU + quantize dh1/dh3", "EC W1/W3",
             "GEMM dX (W1 + W3)", "GEMM dW1 + dW3"]
# with fp16 codes, steps 3 + 4 and 7 + 8 are one launch each (their time lands on 3 and 7)


@dataclass
class FFNOperands:
    """Saved forward state of a SwiGLU FFN block, on the device."""
    X8: torch.Tensor
    s_x: torch.Tensor
    A8: torch.Tensor
    s_a: torch.Tensor
    W1_8: torch.Tensor
    s_w1: torch.Tensor
    W3_8: torch.Tensor
    s_w3: torch.Tensor
    W2_8: torch.Tensor
    s_w2: torch.Tensor
    h1: torch.Tensor
    h3: torch.Tensor


def ffn_forward_operands(X, W1, W3, W2, a, h1, h3, stream=None, code_format=DEFAULT_CODES) -> FFNOperands:
    """RTNE forward operands (per-token scales for X and a, per-output-channel
    scales for the weights) computed with rtne_quantize."""
    cf = code_format
    X8, s_x = rtne_quantize(X, AXIS_ROW, stream=stream, code_format=cf)
    A8, s_a = rtne_quantize(a, AXIS_ROW, stream=stream, code_format=cf)
    W1_8, s_w1 = rtne_quantize(W1, AXIS_COL, stream=stream, code_format=cf)
    W3_8, s_w3 = rtne_quantize(W3, AXIS_COL, stream=stream, code_format=cf)
    W2_8, s_w2 = rtne_quantize(W2, AXIS_COL, stream=stream, code_format=cf)
    return FFNOperands(X8, s_x, A8, s_a, W1_8, s_w1, W3_8, s_w3, W2_8, s_w2, h1, h3)


def ffn_workspace_size(T, d, F, S, round_mode=ROUND_S3R, ec_mode=EC_TWO_WAY, code_format=DEFAULT_CODES,
                       flags=0) -> int:
    return int(lib().s3r_ffn_workspace_size_flags(T, d, F, S, round_mode, ec_mode, code_format, flags))


def grouped_workspace_size(group_offsets, d, F, round_mode=ROUND_S3R, ec_mode=EC_TWO_WAY,
                           code_format=DEFAULT_CODES, flags=0) -> int:
    offs = [int(o) for o in group_offsets]
    arr = (C.c_int64 * len(offs))(*offs)
    return int(lib().s3r_ffn_grouped_workspace_size_flags(C.cast(arr, _VP), len(offs) - 1, d, F, round_mode,
                                                          ec_mode, code_format, flags))


@dataclass
class FFNGrads:
    dX: torch.Tensor
    dW1: torch.Tensor
    dW3: torch.Tensor
    dW2: torch.Tensor


def alloc_ffn_grads(T, d, F, device="cuda") -> FFNGrads:
    f = lambda *s: torch.empty(s, dtype=torch.float32, device=device)
    return FFNGrads(f(T, d), f(d, F), f(d, F), f(F, d))


def moe_forward_operands(X, W1, W3, W2, a, h1, h3, stream=None, code_format=DEFAULT_CODES) -> FFNOperands:
    """Grouped mode: RTNE operands of the expert-sorted routed rows (per-row
    scales) and of every expert's stacked weights W1, W3 [E, d, F], W2 [E, F, d]
    (per-output-channel scales within each expert)."""
    cf = code_format
    X8, s_x = rtne_quantize(X, AXIS_ROW, stream=stream, code_format=cf)
    A8, s_a = rtne_quantize(a, AXIS_ROW, stream=stream, code_format=cf)
    out = []
    for Wk in (W1, W3, W2):
        codes, scales = zip(*[rtne_quantize(Wk[e], AXIS_COL, stream=stream, code_format=cf)
                              for e in range(Wk.shape[0])])
        out += [torch.stack(codes), torch.stack(scales)]
    return FFNOperands(X8, s_x, A8, s_a, *out, h1, h3)


def alloc_moe_grads(R, E, d, F, device="cuda") -> FFNGrads:
    f = lambda *s: torch.empty(s, dtype=torch.float32, device=device)
    return FFNGrads(f(R, d), f(E, d, F), f(E, d, F), f(E, F, d))


def ffn_backward(ops: FFNOperands, dY, S, round_mode=ROUND_S3R, ec_mode=EC_TWO_WAY, seed=0,
                 grads: FFNGrads | None = None, workspace=None, status=None, stream=None,
                 step_events=None, group_offsets=None, fuse_glue=False, widen_codes=False,
                 recompute_a=False) -> FFNGrads:
    """step_events: optional list of FFN_NUM_EVENTS torch.cuda.Event (timing).
    group_offsets: grouped (mixture-of-experts) mode, a list of E + 1 row
    offsets of the expert-sorted rows; the weights in `ops` are then stacked
    per expert and S is ignored.  fuse_glue: run the SwiGLU glue and the
    quantization of dh1, dh3 inside the dA GEMM's epilogue (S3R_FFN_FUSE_GLUE;
    dense block with fp16 codes, not independent SR; dA is then not kept).
    widen_codes: int8 operand codes in `ops` run as fp16 codes (S3R_CODES_S8_F16:
    widened inside the call, results equal to the fp16-code call).
    recompute_a: the call forms the codes of a and their scales from h1 and h3
    (S3R_FFN_RECOMPUTE_A); ops.A8 and ops.s_a are then not used (may be None)."""
    T, d = dY.shape
    F = ops.h1.shape[1]
    dev = dY.device
    fmt = code_format_of(ops.X8)
    flags = (FFN_FUSE_GLUE if fuse_glue else 0) | (FFN_RECOMPUTE_A if recompute_a else 0)
    a8, s_a = (None, None) if recompute_a else (ops.A8, ops.s_a)
    if widen_codes:
        if fmt != CODES_S8:
            raise ValueError("widen_codes takes int8 operand codes")
        fmt = CODES_S8_F16
    if group_offsets is not None:
        offs = [int(o) for o in group_offsets]
        E = len(offs) - 1
        tmax = max([b - a for a, b in zip(offs[:-1], offs[1:])] + [1])
        if grads is None:
            grads = alloc_moe_grads(T, E, d, F, dev)
        need = grouped_workspace_size(offs, d, F, round_mode, ec_mode, fmt, flags)
        S = 0
    else:
        if grads is None:
            grads = alloc_ffn_grads(T, d, F, dev)
        need = ffn_workspace_size(T, d, F, S, round_mode, ec_mode, fmt, flags)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    p = lambda t: None if t is None else t.data_ptr()
    args = _FfnArgs(T, d, F, S, p(_bits(dY)), p(_bits(ops.h1)), p(_bits(ops.h3)), p(ops.X8), p(ops.s_x), p(a8),
                    p(s_a), p(ops.W1_8), p(ops.s_w1), p(ops.W3_8), p(ops.s_w3), p(ops.W2_8), p(ops.s_w2),
                    round_mode, ec_mode, fmt, seed, p(grads.dX), p(grads.dW1), p(grads.dW3), p(grads.dW2),
                    p(workspace), workspace.numel(), p(status), None)
    args.flags = flags
    if group_offsets is not None:
        off_arr = (C.c_int64 * len(offs))(*offs)   # kept alive until the call returns
        args.num_groups = len(offs) - 1
        args.group_offsets = C.cast(off_arr, C.POINTER(C.c_int64))
    if step_events is not None:
        assert len(step_events) == FFN_NUM_EVENTS
        handles = (C.c_void_p * FFN_NUM_EVENTS)(*[C.c_void_p(e.cuda_event) for e in step_events])
        args.step_events = C.cast(handles, C.POINTER(C.c_void_p))
    _check(lib().ffn_backward(C.byref(args), _stream(stream)), "ffn_backward")
    return grads


FFN_WS_VIEWS = ("Q2", "scale2", "Q1", "scale1", "Q3", "scale3", "dA")


def ffn_workspace_views(workspace, T, d, F, S, round_mode=ROUND_S3R, code_format=DEFAULT_CODES, group_offsets=None,
                        group=0) -> dict:
    """Views into an ffn_backward workspace (after the call): the codes and tile
    scales of the three quantized gradients and dA, as laid out by the library
    (s3r_ffn_workspace_offsets).  Grouped mode: the block of expert `group`."""
    assert workspace.dtype == torch.uint8 and workspace.data_ptr() % 256 == 0
    out = (C.c_size_t * 7)()
    if group_offsets is not None:
        offs = [int(o) for o in group_offsets]
        arr = (C.c_int64 * len(offs))(*offs)
        T = offs[group + 1] - offs[group]
        S = T
        _check(lib().s3r_ffn_workspace_offsets(0, d, F, 0, round_mode, code_format, C.cast(arr, _VP), len(offs) - 1,
                                               group, C.cast(out, _VP)), "s3r_ffn_workspace_offsets")
    else:
        _check(lib().s3r_ffn_workspace_offsets(T, d, F, S, round_mode, code_format, None, 0, 0, C.cast(out, _VP)),
               "s3r_ffn_workspace_offsets")
    cdt = _CODE_DTYPE[code_format]
    shapes = {"Q2": ((T, d), cdt), "scale2": ((_cdiv(T, TILE), _cdiv(d, TILE)), torch.float32),
              "Q1": ((T, F), cdt), "scale1": ((_cdiv(T, TILE), _cdiv(F, TILE)), torch.float32),
              "Q3": ((T, F), cdt), "scale3": ((_cdiv(T, TILE), _cdiv(F, TILE)), torch.float32),
              "dA": ((T, F), torch.float32)}
    views = {}
    for i, name in enumerate(FFN_WS_VIEWS):
        shape, dt = shapes[name]
        nbytes = shape[0] * shape[1] * torch.empty(0, dtype=dt).element_size()
        off = int(out[i])
        assert off + nbytes <= workspace.numel(), name
        views[name] = workspace[off:off + nbytes].view(dt).view(shape)
    return views
