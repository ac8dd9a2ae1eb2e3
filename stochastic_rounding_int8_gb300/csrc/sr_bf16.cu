// sr_bf16.cu -- stochastic rounding of fp32 to bf16 and to FP8 e4m3 with
// S3R's shared thresholds, on the hardware stochastic-rounding conversions.
//
// Paper: "Efficient Quantization Training with Stochastic Rounding via
// Structured Subspace Randomness" §II (Blackwell converts to floating-point
// formats with stochastic rounding from random bits the program supplies),
// §III-B (one threshold per token, shared by all its channels).
//
// cvt.rs.satfinite.bf16x2.f32 adds a 16-bit random value to the 16 bits of
// the fp32 magnitude that bf16 drops and truncates; the first source lands
// in the upper half of the result and takes the upper 16 random bits.  With
// random bits 0xFFFF - v the magnitude moves up one bf16 step exactly when
// the dropped bits exceed v: the rounding of a 16-bit threshold v.  S3R's
// v is the upper 16 bits of the token's Philox word (the INT8 quantizer's
// 24-bit threshold, truncated), so all channels of a token share it.
//
// cvt.rs.satfinite.e4m3x4.f32 d, {a, b, c, e}, rbits puts a in byte 3 ... e
// in byte 0; b takes rbits[31:16] and e rbits[15:0] the same way (the e4m3
// magnitude moves up one step iff floor(p 2^16) + r >= 2^16, p its position
// between the two neighbours), while a and c take those 16 bits reversed.
// One threshold per token therefore goes through lanes b and e only (a and
// c carry zeros): two values per conversion.
//
// Streaming kernels: a block takes (row, 8192-column chunk) units; each
// thread converts four groups of 8 values (two 16-byte loads, one 16- or
// 8-byte store).
#include <cuda_bf16.h>

#include "common.cuh"

namespace s3r {
namespace {

enum SrMode { kSrRTNE = 0, kSrS3R = 1, kSrINDEP = 2 };
constexpr int kSrThreads = 256, kSrGroups = 4;
constexpr int64_t kSrChunk = (int64_t)kSrThreads * kSrGroups * 8;   // columns per unit

// Two values, lo in the lower half of the result; v_lo / v_hi their thresholds.
__device__ __forceinline__ uint32_t cvt_rs_pair(float lo, float hi, uint32_t v_lo, uint32_t v_hi) {
    const uint32_t rbits = ((0xFFFFu - v_hi) << 16) | (0xFFFFu - v_lo);
    uint32_t d;
    asm("cvt.rs.satfinite.bf16x2.f32 %0, %1, %2, %3;" : "=r"(d) : "f"(hi), "f"(lo), "r"(rbits));
    return d;
}

// e4m3: lo -> byte 0 (lane e), hi -> byte 2 (lane b) of the result.
__device__ __forceinline__ uint32_t cvt_rs_e4m3_pair(float lo, float hi, uint32_t v_lo, uint32_t v_hi) {
    const uint32_t rbits = ((0xFFFFu - v_hi) << 16) | (0xFFFFu - v_lo);
    uint32_t d;
    asm("cvt.rs.satfinite.e4m3x4.f32 %0, {%1, %2, %3, %4}, %5;"
        : "=r"(d)
        : "f"(0.0f), "f"(hi), "f"(0.0f), "f"(lo), "r"(rbits));
    return d;
}
// e4m3 round to nearest even: lo -> byte 0, hi -> byte 1.
__device__ __forceinline__ uint32_t rn_e4m3_pair(float lo, float hi) {
    unsigned short d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ uint32_t rn_pair(float lo, float hi) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&p);
}

// Thresholds of the 8 elements e0 .. e0 + 7 under independent SR (word e mod 4
// of Philox(e / 4), upper 16 bits).
__device__ __forceinline__ void element_v8(uint64_t e0, uint32_t seed_lo, uint32_t tid, uint32_t (&v)[8]) {
    if ((e0 & 3) == 0) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint64_t c = (e0 >> 2) + h;
            const Philox4 w = philox4x32_10((uint32_t)c, (uint32_t)(c >> 32), 0u, 0u, seed_lo, tid);
            v[4 * h] = w.x >> 16;
            v[4 * h + 1] = w.y >> 16;
            v[4 * h + 2] = w.z >> 16;
            v[4 * h + 3] = w.w >> 16;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint64_t e = e0 + i, c = e >> 2;
            const Philox4 w = philox4x32_10((uint32_t)c, (uint32_t)(c >> 32), 0u, 0u, seed_lo, tid);
            const uint32_t x = (e & 3) == 0 ? w.x : (e & 3) == 1 ? w.y : (e & 3) == 2 ? w.z : w.w;
            v[i] = x >> 16;
        }
    }
}

template <int MODE>
__global__ void __launch_bounds__(kSrThreads) sr_bf16_kernel(const float* X, int64_t N, int64_t ldx, uint16_t* Y,
                                                             int64_t ldy, uint32_t seed_lo, uint32_t tid,
                                                             int64_t units, int64_t upr, bool vec) {
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        const int64_t t = u / upr, c_base = (u - t * upr) * kSrChunk;
        uint32_t vt = 0u;
        if (MODE == kSrS3R) vt = philox4x32_10((uint32_t)t, (uint32_t)(t >> 32), 0u, 0u, seed_lo, tid).x >> 16;
        const float* xr = X + t * ldx;
        uint16_t* yr = Y + t * ldy;
#pragma unroll
        for (int k = 0; k < kSrGroups; ++k) {
            const int64_t c = c_base + 8 * ((int64_t)threadIdx.x + kSrThreads * k);
            if (c >= N) break;
            uint32_t v[8];
            if (MODE == kSrINDEP) element_v8((uint64_t)t * (uint64_t)N + (uint64_t)c, seed_lo, tid, v);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (MODE == kSrS3R) v[i] = vt;
            if (vec && c + 8 <= N) {
                const float4 a = __ldg(reinterpret_cast<const float4*>(xr + c));
                const float4 b = __ldg(reinterpret_cast<const float4*>(xr + c + 4));
                const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                uint32_t w[4];
#pragma unroll
                for (int p = 0; p < 4; ++p)
                    w[p] = MODE == kSrRTNE ? rn_pair(x[2 * p], x[2 * p + 1])
                                         : cvt_rs_pair(x[2 * p], x[2 * p + 1], v[2 * p], v[2 * p + 1]);
                *reinterpret_cast<uint4*>(yr + c) = make_uint4(w[0], w[1], w[2], w[3]);
            } else {
                for (int i = 0; i < 8 && c + i < N; ++i) {
                    const float x = xr[c + i];
                    const uint32_t w = MODE == kSrRTNE ? rn_pair(x, 0.0f) : cvt_rs_pair(x, 0.0f, v[i], 0u);
                    yr[c + i] = (uint16_t)(w & 0xFFFFu);
                }
            }
        }
    }
}

// Four e4m3 codes (values 4 p .. 4 p + 3 of the group) in one 32-bit word.
template <int MODE>
__device__ __forceinline__ uint32_t e4m3_quad(const float (&y)[8], const uint32_t (&v)[8], int p) {
    if (MODE == kSrRTNE)
        return rn_e4m3_pair(y[4 * p], y[4 * p + 1]) | (rn_e4m3_pair(y[4 * p + 2], y[4 * p + 3]) << 16);
    const uint32_t d0 = cvt_rs_e4m3_pair(y[4 * p], y[4 * p + 1], v[4 * p], v[4 * p + 1]);
    const uint32_t d1 = cvt_rs_e4m3_pair(y[4 * p + 2], y[4 * p + 3], v[4 * p + 2], v[4 * p + 3]);
    return __byte_perm(d0, d1, 0x6420);   // bytes 0, 2 of d0, then bytes 0, 2 of d1
}

template <int MODE>
__global__ void __launch_bounds__(kSrThreads) sr_fp8_kernel(const float* X, int64_t N, int64_t ldx, float inv_scale,
                                                            uint8_t* Y, int64_t ldy, uint32_t seed_lo, uint32_t tid,
                                                            int64_t units, int64_t upr, bool vec) {
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        const int64_t t = u / upr, c_base = (u - t * upr) * kSrChunk;
        uint32_t vt = 0u;
        if (MODE == kSrS3R) vt = philox4x32_10((uint32_t)t, (uint32_t)(t >> 32), 0u, 0u, seed_lo, tid).x >> 16;
        const float* xr = X + t * ldx;
        uint8_t* yr = Y + t * ldy;
#pragma unroll
        for (int k = 0; k < kSrGroups; ++k) {
            const int64_t c = c_base + 8 * ((int64_t)threadIdx.x + kSrThreads * k);
            if (c >= N) break;
            uint32_t v[8];
            if (MODE == kSrINDEP) element_v8((uint64_t)t * (uint64_t)N + (uint64_t)c, seed_lo, tid, v);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (MODE != kSrINDEP) v[i] = vt;
            if (vec && c + 8 <= N) {
                const float4 a = __ldg(reinterpret_cast<const float4*>(xr + c));
                const float4 b = __ldg(reinterpret_cast<const float4*>(xr + c + 4));
                const float y[8] = {__fmul_rn(a.x, inv_scale), __fmul_rn(a.y, inv_scale), __fmul_rn(a.z, inv_scale),
                                    __fmul_rn(a.w, inv_scale), __fmul_rn(b.x, inv_scale), __fmul_rn(b.y, inv_scale),
                                    __fmul_rn(b.z, inv_scale), __fmul_rn(b.w, inv_scale)};
                *reinterpret_cast<uint2*>(yr + c) = make_uint2(e4m3_quad<MODE>(y, v, 0), e4m3_quad<MODE>(y, v, 1));
            } else {
                for (int i = 0; i < 8 && c + i < N; ++i) {
                    const float y = __fmul_rn(xr[c + i], inv_scale);
                    const uint32_t w = MODE == kSrRTNE ? rn_e4m3_pair(y, 0.0f) : cvt_rs_e4m3_pair(y, 0.0f, v[i], 0u);
                    yr[c + i] = (uint8_t)(w & 0xFFu);
                }
            }
        }
    }
}

int sm_count_sr() { return s3r_sm_count(); }

}  // namespace
}  // namespace s3r

using namespace s3r;

extern "C" int s3r_sr_bf16(const float* X, int64_t T, int64_t N, int64_t ldx, int round_mode, uint64_t seed,
                           uint32_t tensor_id, void* Y, int64_t ldy, cudaStream_t stream) {
    if (T < 0 || N < 0) return S3R_ERR_ARG;
    if (round_mode != S3R_ROUND_S3R && round_mode != S3R_ROUND_INDEP && round_mode != S3R_ROUND_RTNE)
        return S3R_ERR_ARG;
    if (T == 0 || N == 0) return S3R_OK;
    if (!X || !Y) return S3R_ERR_ARG;
    if (ldx < N || ldy < N) return S3R_ERR_SHAPE;
    const bool vec = s3r_aligned16(X) && s3r_aligned16(Y) && ldx % 4 == 0 && ldy % 8 == 0;
    const int64_t upr = s3r_cdiv(N, kSrChunk), units = T * upr;
    const int64_t cap = (int64_t)sm_count_sr() * 8;
    const unsigned grid = (unsigned)(units < cap ? units : cap);
    uint16_t* y = static_cast<uint16_t*>(Y);
    const uint32_t s = (uint32_t)seed;
    switch (round_mode) {
        case S3R_ROUND_S3R:
            sr_bf16_kernel<kSrS3R><<<grid, kSrThreads, 0, stream>>>(X, N, ldx, y, ldy, s, tensor_id, units, upr, vec);
            break;
        case S3R_ROUND_INDEP:
            sr_bf16_kernel<kSrINDEP><<<grid, kSrThreads, 0, stream>>>(X, N, ldx, y, ldy, s, tensor_id, units, upr, vec);
            break;
        default:
            sr_bf16_kernel<kSrRTNE><<<grid, kSrThreads, 0, stream>>>(X, N, ldx, y, ldy, s, tensor_id, units, upr, vec);
    }
    S3R_CHECK_LAUNCH();
    return S3R_OK;
}

extern "C" int s3r_sr_fp8(const float* X, int64_t T, int64_t N, int64_t ldx, float inv_scale, int round_mode,
                          uint64_t seed, uint32_t tensor_id, void* Y, int64_t ldy, cudaStream_t stream) {
    if (T < 0 || N < 0) return S3R_ERR_ARG;
    if (round_mode != S3R_ROUND_S3R && round_mode != S3R_ROUND_INDEP && round_mode != S3R_ROUND_RTNE)
        return S3R_ERR_ARG;
    if (!(inv_scale > 0.0f) || !(inv_scale <= 3.402823466e38f)) {   // rejects 0, negatives, NaN and infinity
        s3r_record_error("s3r_sr_fp8", "inv_scale must be finite and greater than zero");
        return S3R_ERR_ARG;
    }
    if (T == 0 || N == 0) return S3R_OK;
    if (!X || !Y) return S3R_ERR_ARG;
    if (ldx < N || ldy < N) return S3R_ERR_SHAPE;
    const bool vec = s3r_aligned16(X) && ((uintptr_t)Y & 7u) == 0 && ldx % 4 == 0 && ldy % 8 == 0;
    const int64_t upr = s3r_cdiv(N, kSrChunk), units = T * upr;
    const int64_t cap = (int64_t)sm_count_sr() * 8;
    const unsigned grid = (unsigned)(units < cap ? units : cap);
    uint8_t* y = static_cast<uint8_t*>(Y);
    const uint32_t s = (uint32_t)seed;
    switch (round_mode) {
        case S3R_ROUND_S3R:
            sr_fp8_kernel<kSrS3R><<<grid, kSrThreads, 0, stream>>>(X, N, ldx, inv_scale, y, ldy, s, tensor_id, units,
                                                                    upr, vec);
            break;
        case S3R_ROUND_INDEP:
            sr_fp8_kernel<kSrINDEP><<<grid, kSrThreads, 0, stream>>>(X, N, ldx, inv_scale, y, ldy, s, tensor_id,
                                                                      units, upr, vec);
            break;
        default:
            sr_fp8_kernel<kSrRTNE><<<grid, kSrThreads, 0, stream>>>(X, N, ldx, inv_scale, y, ldy, s, tensor_id, units,
                                                                     upr, vec);
    }
    S3R_CHECK_LAUNCH();
    return S3R_OK;
}
