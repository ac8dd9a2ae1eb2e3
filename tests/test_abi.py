"""The C-ABI library builds, loads and exports every entry point the header
declares; host-side argument checks work without a GPU (nothing is launched
when they fail)."""
import ctypes as C

import pytest

import stochastic_rounding_int8_gb300 as s3r
from stochastic_rounding_int8_gb300 import build as s3r_build


@pytest.fixture(scope="module")
def L():
    s3r_build.build()
    return s3r.lib()


def test_header_declares_the_boundary():
    names = set(s3r.header_functions())
    for want in ["s3r_quantize", "indep_sr_quantize", "rtne_quantize", "s3r_ec_correct", "int8_gemm_dx",
                 "int8_gemm_dw", "ffn_backward", "swiglu_quantize", "s3r_status_string"]:
        assert want in names


def test_library_exports_every_header_symbol(L):
    for name in s3r.header_functions():
        assert hasattr(L, name), name
        assert name in s3r._SIGS, f"binding has no signature for {name}"


def test_status_strings(L):
    assert s3r.status_string(0) == "S3R_OK"
    for code in range(-1, -9, -1):
        assert s3r.status_string(code).startswith("S3R_ERR_")
    assert s3r.status_string(-99) == "S3R_ERR_UNKNOWN"
    assert L.s3r_abi_version() == 104


def test_host_argument_checks_need_no_gpu(L):
    null = None
    P = C.c_void_p(16)
    # null outputs -> S3R_ERR_ARG before any launch
    assert L.s3r_quantize(P, 4, 4, 4, null, null, 0, 0, null, 0, null, null, null, null, null) == -1
    # empty tensors are a no-op
    assert L.s3r_quantize(null, 0, 0, 0, null, null, 0, 0, null, 0, null, null, null, null, null) == 0
    # ldg < N
    assert L.s3r_quantize(P, 4, 8, 4, null, null, 0, 0, P, 0, P, null, null, null, null) == -3
    # unknown code format
    assert L.s3r_quantize(P, 4, 8, 8, null, null, 0, 0, P, 7, P, null, null, null, null) == -1
    # unknown enum values
    assert L.rtne_quantize(P, 4, 4, 4, null, null, 7, P, 0, P, null, null) == -1
    # T not a multiple of S in the correction
    assert L.s3r_ec_correct(P, P, 10, 4, 3, null, 0, null, 0, 0, P, P, P, null, null, null, null, null, 0, null,
                            null) == -3
    # S8 dW workspace too small
    assert L.int8_gemm_dw(P, P, P, 0, 256, 64, 64, null, 0, null, null, null, null, 256, P, P, 8, null, null) == -7
    # mixed or unknown formats in the GEMMs
    assert L.int8_gemm_dx(P, P, P, 5, 4, 16, 4, null, 0, null, null, null, 4, P, 0, null, null) == -1
    # fp16-carried codes need rows of a multiple of 8 codes (TMA strides)
    assert L.int8_gemm_dx(P, P, P, 1, 4, 12, 4, null, 0, null, null, null, 4, P, 0, null, null) == -2


def test_workspace_sizes_are_host_only(L):
    assert L.s3r_ffn_workspace_size(256, 128, 384, 128, 1, 2, 1) > 0
    assert L.s3r_ffn_workspace_size(256, 128, 384, 100, 1, 2, 1) == 0   # T % S != 0
    big_f16 = L.s3r_ffn_workspace_size(8192, 2048, 5632, 2048, 1, 2, 1)
    big_s8 = L.s3r_ffn_workspace_size(8192, 2048, 5632, 2048, 1, 2, 0)
    assert big_f16 > big_s8 - 200 * 2 ** 20   # fp16 codes double Q; S8 adds the dW transposes
    assert L.int8_gemm_dw_workspace_size(300, 5, 7, 0) >= (5 + 7) * 304
    assert L.int8_gemm_dw_workspace_size(300, 5, 7, 1) == 0
    assert L.s3r_ec_workspace_size(0, 5) == 0


def _header_struct_fields(name):
    import re
    txt = open(s3r.HEADER).read()
    body = re.search(r"struct " + name + r" \{(.*?)\};", txt, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = []
    for decl in body.split(";"):
        decl = decl.strip()
        if not decl:
            continue
        for part in re.split(r",", decl):
            fields.append(re.findall(r"\w+", part)[-1])
    return fields


def test_ffn_args_struct_layout_matches_header():
    """The ctypes mirrors of struct s3r_ffn_args and struct s3r_ffn_fwd_args
    have one field per header field, in order."""
    assert _header_struct_fields("s3r_ffn_args") == [f for f, _ in s3r._FfnArgs._fields_]
    assert _header_struct_fields("s3r_ffn_fwd_args") == [f for f, _ in s3r._FfnFwdArgs._fields_]


def test_forward_and_sr_bf16_arguments_checked_on_host(L):
    """Host-side checks of the forward and SR-to-bf16 entries (fake,
    never-dereferenced pointers; no launch happens)."""
    import ctypes as C
    fake = C.c_void_p(0x1000)
    S3R_ERR_ARG, S3R_ERR_SHAPE, S3R_ERR_UNSUPPORTED = -1, -3, -8
    # int8-carried codes are not taken by the forward
    assert L.int8_gemm_fwd(fake, fake, fake, fake, s3r.CODES_S8, 8, 16, 16, fake, None, None) == S3R_ERR_UNSUPPORTED
    assert L.int8_gemm_fwd(fake, fake, fake, fake, s3r.CODES_F16, -1, 16, 16, fake, None, None) == S3R_ERR_ARG
    assert L.int8_gemm_fwd(fake, fake, fake, fake, s3r.CODES_F16, 0, 16, 16, fake, None, None) == 0
    assert L.int8_gemm_fwd_swiglu(fake, fake, fake, fake, None, None, s3r.CODES_F16, 8, 16, 16, fake, fake, None,
                                  None, None) == S3R_ERR_ARG   # W3 missing
    assert L.swiglu_fwd_quantize(fake, fake, 4, 16, 8, None, fake, s3r.CODES_F16, fake, None, None) == S3R_ERR_SHAPE
    assert L.swiglu_fwd_quantize(fake, fake, 4, 16, 16, None, fake, 7, fake, None, None) == S3R_ERR_ARG
    assert L.s3r_sr_bf16(fake, 4, 16, 8, s3r.ROUND_S3R, 0, 0, fake, 16, None) == S3R_ERR_SHAPE
    assert L.s3r_sr_bf16(fake, 4, 16, 16, s3r.ROUND_S3R_7BIT, 0, 0, fake, 16, None) == S3R_ERR_ARG
    assert L.s3r_sr_bf16(fake, 0, 16, 16, s3r.ROUND_S3R, 0, 0, fake, 16, None) == 0
    args = s3r._FfnFwdArgs(8, 16, 16, fake, fake, fake, fake, 1, s3r.CODES_S8)
    assert L.ffn_forward(C.byref(args), None) == S3R_ERR_UNSUPPORTED


def test_grouped_args_rejected_on_host():
    """Grouped-mode offsets are checked before any launch: they must start at
    0, end at T and never decrease (fake, never-dereferenced pointers)."""
    import ctypes as C
    fake = C.c_void_p(0x1000)
    for offs, T in (([0, 5, 9], 10), ([1, 5, 10], 10), ([0, 6, 4, 10], 10)):
        arr = (C.c_int64 * len(offs))(*offs)
        a = s3r._FfnArgs(T, 64, 128, 0, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                         s3r.ROUND_S3R, s3r.EC_TWO_WAY, s3r.CODES_F16, 0, fake, fake, fake, fake, fake, 1 << 30,
                         None, None, len(offs) - 1, C.cast(arr, C.POINTER(C.c_int64)))
        assert s3r.lib().ffn_backward(C.byref(a), None) == -1


def test_sr_fp8_rejects_bad_scales_on_host(L):
    """s3r_sr_fp8 takes only a finite scale above zero; zero, negative, NaN and
    infinite scales are rejected before any launch (fake pointers)."""
    fake = C.c_void_p(0x1000)
    for bad in (0.0, -1.0, -0.0, float("nan"), float("inf"), float("-inf")):
        assert L.s3r_sr_fp8(fake, 4, 16, 16, bad, s3r.ROUND_S3R, 0, 0, fake, 16, None) == -1, bad
        assert "inv_scale" in L.s3r_last_error().decode()
    assert L.s3r_sr_fp8(fake, 0, 16, 16, 0.5, s3r.ROUND_S3R, 0, 0, fake, 16, None) == 0   # empty: no launch


def test_ffn_workspace_offsets(L):
    """The inspection hook lays its views inside the workspace, without overlap,
    in dense and grouped mode; grouped blocks follow each other."""
    out = (C.c_size_t * 7)()
    T, d, F, S = 512, 136, 392, 256
    assert L.s3r_ffn_workspace_offsets(T, d, F, S, 1, 1, None, 0, 0, C.cast(out, C.c_void_p)) == 0
    cd = 2
    sizes = [T * d * cd, 4 * 2 * 2, T * F * cd, 4 * 4 * 4, T * F * cd, 4 * 4 * 4, T * F * 4]
    spans = sorted((int(o), int(o) + n) for o, n in zip(out, sizes))
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))
    assert spans[-1][1] <= L.s3r_ffn_workspace_size(T, d, F, S, 1, 2, 1)
    assert all(int(o) % 256 == 0 for o in out)
    offs = [0, 300, 300, 812]
    arr = (C.c_int64 * 4)(*offs)
    g0 = (C.c_size_t * 7)()
    g2 = (C.c_size_t * 7)()
    assert L.s3r_ffn_workspace_offsets(0, d, F, 0, 1, 1, C.cast(arr, C.c_void_p), 3, 0, C.cast(g0, C.c_void_p)) == 0
    assert L.s3r_ffn_workspace_offsets(0, d, F, 0, 1, 1, C.cast(arr, C.c_void_p), 3, 2, C.cast(g2, C.c_void_p)) == 0
    first = L.s3r_ffn_workspace_size(300, d, F, 300, 1, 2, 1)
    assert int(g2[0]) - int(g0[0]) >= first - 256
    assert int(g2[6]) + 512 * F * 4 <= L.s3r_ffn_grouped_workspace_size(C.cast(arr, C.c_void_p), 3, d, F, 1, 2, 1)
    # the empty expert has no block
    assert L.s3r_ffn_workspace_offsets(0, d, F, 0, 1, 1, C.cast(arr, C.c_void_p), 3, 1, C.cast(g0, C.c_void_p)) == -1


def test_widened_codes_workspace_and_checks(L):
    """S3R_CODES_S8_F16 (int8 operand codes widened inside ffn_backward): its
    workspace is the fp16 block's plus the five fp16 copies, its intermediates
    sit where the fp16 block keeps them, and its own checks run before any
    launch (fake, never-dereferenced pointers)."""
    r = lambda b: (b + 255) // 256 * 256
    T, d, F, S = 512, 136, 392, 256
    f16 = L.s3r_ffn_workspace_size(T, d, F, S, 1, 2, s3r.CODES_F16)
    wide = L.s3r_ffn_workspace_size(T, d, F, S, 1, 2, s3r.CODES_S8_F16)
    assert wide == f16 + 255 + r(2 * T * d) + r(2 * T * F) + 3 * r(2 * d * F)
    offs = [0, 300, 300, 812]
    arr = (C.c_int64 * 4)(*offs)
    g16 = L.s3r_ffn_grouped_workspace_size(C.cast(arr, C.c_void_p), 3, d, F, 1, 2, s3r.CODES_F16)
    gw = L.s3r_ffn_grouped_workspace_size(C.cast(arr, C.c_void_p), 3, d, F, 1, 2, s3r.CODES_S8_F16)
    assert gw == g16 + 255 + r(2 * 812 * d) + r(2 * 812 * F) + 3 * r(2 * 3 * d * F)
    a, b = (C.c_size_t * 7)(), (C.c_size_t * 7)()
    assert L.s3r_ffn_workspace_offsets(T, d, F, S, 1, s3r.CODES_F16, None, 0, 0, C.cast(a, C.c_void_p)) == 0
    assert L.s3r_ffn_workspace_offsets(T, d, F, S, 1, s3r.CODES_S8_F16, None, 0, 0, C.cast(b, C.c_void_p)) == 0
    assert list(a) == list(b)
    fake = C.c_void_p(0x1000)

    def call(d_, F_, ws_bytes):
        args = s3r._FfnArgs(T, d_, F_, S, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                            fake, s3r.ROUND_S3R, s3r.EC_TWO_WAY, s3r.CODES_S8_F16, 0, fake, fake, fake, fake, fake,
                            ws_bytes, None, None)
        return L.ffn_backward(C.byref(args), None)
    before = L.s3r_kernel_launch_count()
    assert call(132, F, 1 << 40) == -2                # d not a multiple of 8: the fp16 GEMMs' rows
    assert call(d, F, wide - 1) == -7                 # the widened copies do not fit
    assert L.s3r_kernel_launch_count() == before


def test_recompute_a_workspace_and_checks(L):
    """S3R_FFN_RECOMPUTE_A: the workspace adds the recomputed codes of a and
    their scales; A8 and s_a must be NULL with the flag and A8 given without
    it, all checked before any launch (fake, never-dereferenced pointers)."""
    r = lambda b: (b + 255) // 256 * 256
    T, d, F, S = 512, 136, 392, 256
    R = s3r.FFN_RECOMPUTE_A
    for fmt, cs in ((s3r.CODES_F16, 2), (s3r.CODES_S8_F16, 2), (s3r.CODES_S8, 1)):
        base = L.s3r_ffn_workspace_size(T, d, F, S, 1, 2, fmt)
        assert L.s3r_ffn_workspace_size_flags(T, d, F, S, 1, 2, fmt, 0) == base
        assert L.s3r_ffn_workspace_size_flags(T, d, F, S, 1, 2, fmt, R) == base + 255 + r(cs * T * F) + r(4 * T)
    offs = [0, 300, 300, 812]
    arr = (C.c_int64 * 4)(*offs)
    g = L.s3r_ffn_grouped_workspace_size(C.cast(arr, C.c_void_p), 3, d, F, 1, 2, s3r.CODES_F16)
    assert L.s3r_ffn_grouped_workspace_size_flags(C.cast(arr, C.c_void_p), 3, d, F, 1, 2, s3r.CODES_F16, R) == \
        g + 255 + r(2 * 812 * F) + r(4 * 812)
    fake = C.c_void_p(0x1000)
    need = L.s3r_ffn_workspace_size_flags(T, d, F, S, 1, 2, s3r.CODES_F16, R)

    def call(a8, s_a, flags, ws_bytes):
        args = s3r._FfnArgs(T, d, F, S, fake, fake, fake, fake, fake, a8, s_a, fake, fake, fake, fake, fake, fake,
                            s3r.ROUND_S3R, s3r.EC_TWO_WAY, s3r.CODES_F16, 0, fake, fake, fake, fake, fake,
                            ws_bytes, None, None)
        args.flags = flags
        return L.ffn_backward(C.byref(args), None)
    before = L.s3r_kernel_launch_count()
    assert call(fake, None, R, need) == -1        # A8 given with the flag
    assert call(None, fake, R, need) == -1        # s_a given with the flag
    assert call(None, None, 0, need) == -1        # no A8 and no flag
    assert call(None, None, R, need - 1) == -7    # the recomputed codes do not fit
    assert L.s3r_kernel_launch_count() == before
