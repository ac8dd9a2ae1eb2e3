// common.cuh -- device helpers shared by the libs3r kernels (sm_103a).
//
// The library is compiled with -fmad=false: no multiply-add is contracted
// unless written as fmaf(), so every fp32 operation that decides an int8 code
// happens exactly as the header documents it.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/s3r.h"

namespace s3r {

constexpr int kTile = S3R_TILE;

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
// as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies whose high
// halves are xored with the other two counter words and the key; the key is
// bumped by the Weyl increments between rounds.
// ---------------------------------------------------------------------------
struct Philox4 {
    uint32_t x, y, z, w;
};

__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                                 uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo_a = 0xD2511F53u * c0, hi_a = __umulhi(0xD2511F53u, c0);
        const uint32_t lo_b = 0xCD9E8D57u * c2, hi_b = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = hi_b ^ c1 ^ k0;
        const uint32_t n2 = hi_a ^ c3 ^ k1;
        c0 = n0;
        c1 = lo_b;
        c2 = n2;
        c3 = lo_a;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return Philox4{c0, c1, c2, c3};
}

// Top 24 bits of a word as a threshold on the grid {0, 2^-24, ..., 1 - 2^-24}.
__device__ __forceinline__ float unit24(uint32_t w) { return (float)(w >> 8) * 5.9604644775390625e-8f; }

// S3R per-token threshold (Phi_2D): word 0 of Philox(counter = t, key = (seed, id)).
__device__ __forceinline__ float token_threshold(uint64_t t, uint32_t seed_lo, uint32_t tensor_id) {
    return unit24(philox4x32_10((uint32_t)t, (uint32_t)(t >> 32), 0u, 0u, seed_lo, tensor_id).x);
}

// The paper's 7-bit per-token thresholds: four per word (token t takes byte t mod 4
// of word 0 of Philox(counter = t / 4)); its upper 7 bits k give (k + 1/2) / 128,
// the grid shifted by half a step.
__device__ __forceinline__ float token_threshold7(uint64_t t, uint32_t seed_lo, uint32_t tensor_id) {
    const uint64_t c = t >> 2;
    const uint32_t w = philox4x32_10((uint32_t)c, (uint32_t)(c >> 32), 0u, 0u, seed_lo, tensor_id).x;
    const uint32_t k = (w >> (8u * (uint32_t)(t & 3u) + 1u)) & 0x7Fu;
    return ((float)k + 0.5f) * 0.0078125f;   // exact: k + 1/2 has at most 8 significant bits
}

// Phi_bcast: one threshold per example b, word 0 of Philox(counter = (b, 0, 1, 0)).
__device__ __forceinline__ float example_threshold(uint64_t b, uint32_t seed_lo, uint32_t tensor_id) {
    return unit24(philox4x32_10((uint32_t)b, (uint32_t)(b >> 32), 1u, 0u, seed_lo, tensor_id).x);
}

// ---------------------------------------------------------------------------
// bf16 helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t packed) { return __uint_as_float(packed & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_at(const uint16_t* p) { return __uint_as_float((uint32_t)(*p) << 16); }

// ---------------------------------------------------------------------------
// exp by Cody-Waite reduction x = n ln2 + r (ln2 = head + tail, the head with
// 16 significant bits so n*head is exact), e^r by the degree-7 Taylor series
// in Horner form, times 2^n built in the exponent field.  The argument is
// clamped to [-87, 88] so 2^n is a normal number.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float exp_cw(float x) {
    x = fminf(fmaxf(x, -87.0f), 88.0f);
    const float n = rintf(x * 1.44269502162933349609375f);     // log2(e) in fp32
    float r = fmaf(-n, 0.693145751953125f, x);                   // 45426 / 2^16
    r = fmaf(-n, 1.42860682028622683e-06f, r);                   // ln2 - head
    float poly = 1.98412701138295233e-04f;                       // 1/5040
    poly = fmaf(poly, r, 1.38888892251998186e-03f);              // 1/720
    poly = fmaf(poly, r, 8.33333376795053482e-03f);              // 1/120
    poly = fmaf(poly, r, 4.16666679084300995e-02f);              // 1/24
    poly = fmaf(poly, r, 1.66666671633720398e-01f);              // 1/6
    poly = fmaf(poly, r, 0.5f);
    poly = fmaf(poly, r, 1.0f);
    poly = fmaf(poly, r, 1.0f);
    const float two_n = __int_as_float(((int)n + 127) << 23);
    return poly * two_n;
}

__device__ __forceinline__ float sigmoid_cw(float x) { return 1.0f / (1.0f + exp_cw(-x)); }

// ---------------------------------------------------------------------------
// Packed fp32 pair arithmetic (sm_100 family): one instruction per two lanes,
// each rounded to nearest exactly like the scalar operation.  Caution: ptxas
// fuses f2_mul followed by an f2_add / f2_sub that is the product's only use
// into one packed fma despite the .rn qualifiers (measured on sm_103a); where
// the separate rounding matters, do that add with the scalar __fadd_rn.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
    float2 d;
    asm("{\n .reg .b64 x, y, z;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n mul.rn.f32x2 z, x, y;\n"
        " mov.b64 {%0, %1}, z;\n}\n"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 f2_add(float2 a, float2 b) {
    float2 d;
    asm("{\n .reg .b64 x, y, z;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n add.rn.f32x2 z, x, y;\n"
        " mov.b64 {%0, %1}, z;\n}\n"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 f2_sub(float2 a, float2 b) {
    float2 d;
    asm("{\n .reg .b64 x, y, z;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n sub.rn.f32x2 z, x, y;\n"
        " mov.b64 {%0, %1}, z;\n}\n"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
// a * b + c with one rounding per lane
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n .reg .b64 x, y, z, w;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n mov.b64 z, {%6, %7};\n"
        " fma.rn.f32x2 w, x, y, z;\n mov.b64 {%0, %1}, w;\n}\n"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// a + b per lane, rounded toward minus infinity
__device__ __forceinline__ float2 f2_add_rm(float2 a, float2 b) {
    float2 d;
    asm("{\n .reg .b64 x, y, z;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n add.rm.f32x2 z, x, y;\n"
        " mov.b64 {%0, %1}, z;\n}\n"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
// a + b per lane, rounded toward plus infinity
__device__ __forceinline__ float2 f2_add_rp(float2 a, float2 b) {
    float2 d;
    asm("{\n .reg .b64 x, y, z;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n add.rp.f32x2 z, x, y;\n"
        " mov.b64 {%0, %1}, z;\n}\n"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
// a - b per lane, rounded toward plus infinity
__device__ __forceinline__ float2 f2_sub_rp(float2 a, float2 b) {
    float2 d;
    asm("{\n .reg .b64 x, y, z;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n sub.rp.f32x2 z, x, y;\n"
        " mov.b64 {%0, %1}, z;\n}\n"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
// 1.0f if a < b else 0.0f
__device__ __forceinline__ float lt_one(float a, float b) {
    float d;
    asm("set.lt.f32.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}
// per bf16 half: a value whose magnitude is max(|a|, |b|) (NaN if either is NaN); the
// sign bit is the xor of the inputs' and carries no meaning here
__device__ __forceinline__ uint32_t bf16x2_absmax_nan(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// max(m, |a|, |b|), NaN if any of them is NaN
__device__ __forceinline__ float max3_abs_nan(float m, float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(m), "f"(fabsf(a)), "f"(fabsf(b)));
    return d;
}
// 1.5 * 2^23: for |x| < 2^22, x + kMagic lands in [2^23, 2^24), where the
// float spacing is 1, so the add rounds x to an integer (in the add's
// rounding mode) and the low byte of the sum's bits is that integer mod 256.
constexpr float kMagic = 12582912.0f;

// 1 / d correctly rounded for d in [1, 2^126): the hardware approximation
// (within one ulp) refined by one Newton-Raphson step on the residual,
// y + y (1 - d y) with both operations fused (Markstein's correction).  An
// exhaustive GPU comparison over every float in [1, 2^126) found it equal to
// the IEEE reciprocal; larger d (a result below the normal range, where the
// approximation flushes) takes the IEEE reciprocal itself.
static __device__ __noinline__ float2 rcp2_ieee(float2 d) { return make_float2(__frcp_rn(d.x), __frcp_rn(d.y)); }
__device__ __forceinline__ float2 rcp2_den(float2 d) {
    if (fmaxf(d.x, d.y) >= 0x1p126f) return rcp2_ieee(d);
    float2 y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y.x) : "f"(d.x));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y.y) : "f"(d.y));
    const float2 e = f2_fma(make_float2(-d.x, -d.y), y, make_float2(1.0f, 1.0f));
    return f2_fma(e, y, y);
}

// sigmoid_cw of two lanes at once, per lane bit-identical to sigmoid_cw (exp_cw
// of -x, the correctly rounded reciprocal standing for the IEEE quotient
// 1 / (1 + e)).
__device__ __forceinline__ float2 sigmoid2(float2 x) {
    // exp_cw(-x): clamp, n = rint(-x log2 e), r = -x - n ln2 (two parts), Taylor
    const float a0 = fminf(fmaxf(-x.x, -87.0f), 88.0f), a1 = fminf(fmaxf(-x.y, -87.0f), 88.0f);
    const float2 a = make_float2(a0, a1);
    const float2 t = f2_mul(a, make_float2(1.44269502162933349609375f, 1.44269502162933349609375f));
    // n = rint(t) as kMagic + t rounded to nearest, minus kMagic (|t| <= 127); the sum's bits are
    // kMagic's plus n, which gives 2^n without a conversion.  Per-lane adds: a packed add as the
    // product's only use would be fused into an fma.
    const float tm0 = __fadd_rn(t.x, kMagic), tm1 = __fadd_rn(t.y, kMagic);
    const float2 n = f2_sub(make_float2(tm0, tm1), make_float2(kMagic, kMagic));
    float2 r = f2_fma(n, make_float2(-0.693145751953125f, -0.693145751953125f), a);
    r = f2_fma(n, make_float2(-1.42860682028622683e-06f, -1.42860682028622683e-06f), r);
    float2 poly = make_float2(1.98412701138295233e-04f, 1.98412701138295233e-04f);
    poly = f2_fma(poly, r, make_float2(1.38888892251998186e-03f, 1.38888892251998186e-03f));
    poly = f2_fma(poly, r, make_float2(8.33333376795053482e-03f, 8.33333376795053482e-03f));
    poly = f2_fma(poly, r, make_float2(4.16666679084300995e-02f, 4.16666679084300995e-02f));
    poly = f2_fma(poly, r, make_float2(1.66666671633720398e-01f, 1.66666671633720398e-01f));
    poly = f2_fma(poly, r, make_float2(0.5f, 0.5f));
    poly = f2_fma(poly, r, make_float2(1.0f, 1.0f));
    poly = f2_fma(poly, r, make_float2(1.0f, 1.0f));
    // 2^n = (bits(tm) - bits(kMagic) + 127) << 23 (0x4B400000 = bits of kMagic), as one multiply-add
    // on the bits (mod 2^32)
    constexpr uint32_t kExpBias = (uint32_t)(127 - (int)0x4B400000) << 23;
    const float2 two_n = make_float2(__uint_as_float(__float_as_uint(tm0) * 8388608u + kExpBias),
                                     __uint_as_float(__float_as_uint(tm1) * 8388608u + kExpBias));
    // (1 + poly 2^n may fuse into an fma: a product with a power of two is exact.)
    const float2 e = f2_mul(poly, two_n);
    const float2 den = f2_add(make_float2(1.0f, 1.0f), e);
    return rcp2_den(den);
}

// The SwiGLU derivative terms of two lanes at once, per lane bit-identical to
//   s = sigmoid_cw(x); silu = x * s; dsilu = s * (1 + x * (1 - s))
__device__ __forceinline__ void swiglu_terms2(float2 x, float2& silu, float2& dsilu) {
    const float2 s = sigmoid2(x);
    silu = f2_mul(x, s);
    const float2 one = make_float2(1.0f, 1.0f);
    // ptxas contracts a packed multiply whose only use is a packed add into a
    // packed fma, .rn or not; the scalar __fadd_rn is never contracted, so the
    // product x (1 - s) is rounded on its own as the documented order requires.
    const float2 xt = f2_mul(x, f2_sub(one, s));
    dsilu = f2_mul(s, make_float2(__fadd_rn(1.0f, xt.x), __fadd_rn(1.0f, xt.y)));
}

// Tile scale delta = amax / 127 and inv = 127 / amax rounded toward zero (so
// |g * inv| <= 127 and no code leaves [-127, 127]) from the tile absmax bits
// (non-negative floats; NaN and infinity order last).
__device__ __forceinline__ void tile_scales(uint32_t amax_bits, float& d, float& inv) {
    const bool nonfinite = amax_bits >= 0x7F800000u;
    const float amx = __uint_as_float(amax_bits);
    d = nonfinite ? __uint_as_float(0x7FC00000u) : amx / 127.0f;
    inv = (amax_bits == 0u || nonfinite) ? 0.0f : __fdiv_rz(127.0f, amx);
}

// Record a device-side error (first writer wins is not needed: any error code
// tells the caller to look; all writers write a negative constant).
__device__ __forceinline__ void set_status(int* d_status, int code) {
    if (d_status) *(volatile int*)d_status = code;
}

}  // namespace s3r

// Host-side helpers.  Every kernel launch is followed by S3R_CHECK_LAUNCH(),
// which also counts it (s3r_kernel_launch_count()).  Failures are described
// in a thread-local message (s3r_last_error()).
void s3r_count_launch();
void s3r_record_error(const char* where, const char* what);
int s3r_cuda_fail(const char* where, cudaError_t err);
// Streaming multiprocessors of the current device (looked up once per device).
int s3r_sm_count();
// Raises the dynamic shared-memory limit of kernel `func` to `bytes` on the
// current device, once per (kernel, device) pair (the attribute is per
// device); thread-safe.  Returns S3R_OK or S3R_ERR_CUDA (described under `what`).
int s3r_kernel_smem(const void* func, int bytes, const char* what);

// Grouped tcgen05 GEMMs on fp16-carried codes (gemm_umma.cu): up to 24
// problems in one persistent launch, each computed exactly as a
// launch of its own would compute it.
struct UmmaDxProblem {
    const void* Q;               // [T, N] codes, tile scales, W [K, N], correction terms
    const float* tile_scale;
    const void* W;
    const float* eps;
    const int32_t* rowsum;
    const float* v;
    const void* Q3;              // optional second term (NULL: one term)
    const float* tile_scale3;
    const void* W3;
    const float* eps3;
    const int32_t* rowsum3;
    const float* v3;
    int64_t T, N, K;
    const float* s_x;
    int ec_mode;
    int64_t S;
    float* dX;
    int accumulate;
    int32_t* dump;
};
struct UmmaDwProblem {
    const void* X;               // [T, K] codes
    const void* Q;               // [T, N] codes and their tile scales
    const float* tile_scale;
    int64_t T, K, N;
    const float* s_w;
    int ec_mode;
    const float* colmean;
    const float* mu;
    const int32_t* xsum;
    const float* p;
    int64_t S;
    float* dW;
    int32_t* dump;
};
int umma_dx_group(const UmmaDxProblem* probs, int n, int* d_status, cudaStream_t stream);
int umma_dw_group(const UmmaDwProblem* probs, int n, int* d_status, cudaStream_t stream);
// dX and dW problems together (up to 24 in all): one launch, tiles of the
// longest problems first
int umma_mixed_group(const UmmaDxProblem* dx, int ndx, const UmmaDwProblem* dw, int ndw, int* d_status,
                     cudaStream_t stream);
// The SwiGLU glue and the quantization of its two outputs run in the epilogue
// of one dX problem of a mixed launch (the activation gradient dA of the
// block's down projection, one contraction term): instead of storing dA, each
// 128 x 128 quarter-tile becomes dh1 = (dA h3) sigma'(h1), dh3 = dA silu(h1),
// folded with s_x and s_w1 / s_w3, rounded to fp16-carried codes Q1, Q3 with
// their tile scales and error partials -- the same values, bit for bit, as
// swiglu_quantize_ex on the stored dA (the partials up to summation order).
struct UmmaGlue {
    int dx_index;                // which dX problem of the launch carries the glue
    int round_mode;              // S3R_ROUND_S3R, _S3R_7BIT, _BCAST or _RTNE
    uint64_t seed;
    uint32_t tid1, tid3;
    int64_t S;                   // tokens per example (S3R_ROUND_BCAST)
    const void* h1;              // bf16 [T, F], row stride ldh
    const void* h3;
    int64_t ldh;
    const float* s_x;            // folds (NULL: 1)
    const float* s_w1;
    const float* s_w3;
    void* Q1;                    // fp16 codes [T, F]
    void* Q3;
    float* scale1;               // tile scales [ceil(T/128), ceil(F/128)]
    float* scale3;
    float* tok1;                 // per-token error partials [T, ceil(F/128)] (NULL: none)
    float* tok3;
    float* col1;                 // per-channel error partials [ceil(T/128), F]
    float* col3;
};
int umma_mixed_group_glue(const UmmaDxProblem* dx, int ndx, const UmmaDwProblem* dw, int ndw, const UmmaGlue* glue,
                          int* d_status, cudaStream_t stream);
// The INT8 forward on fp16-carried codes: Y = (X W * s_x) * s_w (W3 == NULL),
// or with W3 the gate and up projections through the SwiGLU gate into bf16
// h1, h3 and a (Y unused).  X [T, K], W and W3 [K, N] as stored.
int umma_fwd(const void* X, const float* s_x, const void* W, const float* s_w, const void* W3, const float* s_w3,
             int64_t T, int64_t K, int64_t N, float* Y, uint16_t* h1, uint16_t* h3, uint16_t* a, int* d_status,
             cudaStream_t stream);

// Test hooks of the bounded waits (see s3r_debug_wait_timeout): each runs its
// kernel family's own wait routine on a barrier that nothing arrives on.
int umma_wait_probe(uint64_t limit_ns, int raise_abort, int* d_status, unsigned long long* waited_ns,
                    cudaStream_t stream);
int quant_wait_probe(uint64_t limit_ns, int* d_status, unsigned long long* waited_ns, cudaStream_t stream);
int ec_wait_probe(uint64_t limit_ns, int raise_abort, int* d_status, unsigned long long* waited_ns,
                  cudaStream_t stream);

// S3R-EC factors of the two linears that read the same input X (W1 and W3 of
// the SwiGLU block) in one pass; bit-identical to two s3r_ec_correct calls
// (ec.cu).
size_t s3r_ec_pair_workspace_size(int64_t T, int64_t K);
// max_ctas > 0 caps the grid of the streaming pass (several calls sharing the
// GPU on side streams); 0: all SMs.
int s3r_ec_correct_pair(const float* tok1, const float* col1, const void* W1_8, float* eps1, float* mu1,
                        float* colmean1, int32_t* rowsum1, float* v1, int32_t* xsum1, float* p1, const float* tok3,
                        const float* col3, const void* W3_8, float* eps3, float* mu3, float* colmean3,
                        int32_t* rowsum3, float* v3, int32_t* xsum3, float* p3, int64_t T, int64_t N, int64_t S,
                        int64_t K, const void* X8, int code_format, int ec_mode, void* workspace,
                        size_t workspace_bytes, int max_ctas, int* d_status, cudaStream_t stream);
// s3r_ec_correct with that cap.
int s3r_ec_correct_capped(const float* tok_err_part, const float* col_err_part, int64_t T, int64_t N, int64_t S,
                          const void* W8, int64_t K, const void* X8, int code_format, int ec_mode, float* eps,
                          float* mu, float* colmean, int32_t* rowsum, float* v, int32_t* xsum, float* p,
                          void* workspace, size_t workspace_bytes, int max_ctas, int* d_status,
                          cudaStream_t stream);
#define S3R_CHECK_LAUNCH()                                               \
    do {                                                                 \
        s3r_count_launch();                                              \
        cudaError_t _e = cudaPeekAtLastError();                          \
        if (_e != cudaSuccess) {                                         \
            (void)cudaGetLastError();                                    \
            return s3r_cuda_fail(__FILE__ ":" S3R_STR(__LINE__), _e);    \
        }                                                                \
    } while (0)
#define S3R_STR2(x) #x
#define S3R_STR(x) S3R_STR2(x)

static inline bool s3r_aligned16(const void* p) { return (((uintptr_t)p) & 15u) == 0; }
__host__ __device__ static inline int64_t s3r_cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
