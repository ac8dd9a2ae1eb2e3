// ec.cu -- S3R-EC statistics and correction factors.
//
// Paper: "Efficient Quantization Training with Stochastic Rounding via
// Structured Subspace Randomness" §III-D "Two-way correction": the token
// means eps, the per-example channel means colmean_b and grand mean mu_b form
// the orthogonal projection P(E_b) = 1 colmean_b^T + eps_b 1^T - mu_b 1 1^T;
// its image through the activation-gradient product is eps[t] W1_D + v_b with
// v_b = W8 (colmean_b - mu_b), and through the weight-gradient product
// sum_b xsum_b (colmean_b - mu_b)^T + X8^T eps.
//
// Every reduction runs in a fixed order (no float atomics), so results are
// deterministic run to run.
#include <cuda_fp16.h>

#include "common.cuh"

namespace s3r {

__device__ __forceinline__ int code_value(int8_t c) { return c; }
__device__ __forceinline__ int code_value(__half c) { return __half2int_rn(c); }

// eps[t] = (sum_j tok[t, j]) / N ;  colmean[b, n] = (sum_{tile rows i of b} col[i, n]) / S
__global__ void ec_means_kernel(const float* tok, const float* col, int64_t T, int64_t N, int64_t S, int64_t ntc,
                                int64_t ntr, float* eps, float* colmean) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t B = T / S;
    if (i < T) {
        float s = 0.0f;
        for (int64_t j = 0; j < ntc; ++j) s += tok[i * ntc + j];
        eps[i] = s / (float)N;
    } else if (i < T + B * N) {
        const int64_t k = i - T, b = k / N, n = k % N;
        int64_t r_begin, r_end;
        if (B == 1) { r_begin = 0; r_end = ntr; }
        else { r_begin = b * (S / kTile); r_end = (b + 1) * (S / kTile); }
        float s = 0.0f;
        for (int64_t r = r_begin; r < r_end; ++r) s += col[r * N + n];
        colmean[b * N + n] = s / (float)S;
    }
}

// mu[b] = (1/S) sum_{t in b} eps[t]
__global__ void __launch_bounds__(256) ec_mu_kernel(const float* eps, int64_t S, float* mu) {
    const int64_t b = blockIdx.x;
    __shared__ float red[256];
    float s = 0.0f;
    for (int64_t t = threadIdx.x; t < S; t += 256) s += eps[b * S + t];
    red[threadIdx.x] = s;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) mu[b] = red[0] / (float)S;
}

// One warp per weight row k: rowsum[k] = sum_n W8[k,n]; v[b,k] = sum_n (colmean[b,n]-mu[b]) W8[k,n].
template <typename CodeT>
__global__ void __launch_bounds__(256) ec_gemv_kernel(const CodeT* W8, int64_t K, int64_t N, int64_t B,
                                                      const float* colmean, const float* mu, int32_t* rowsum,
                                                      float* v) {
    const int64_t k = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (k >= K) return;
    const CodeT* w = W8 + k * N;
    int32_t rs = 0;
    for (int64_t n = lane; n < N; n += 32) rs += code_value(w[n]);
    for (int o = 16; o > 0; o >>= 1) rs += __shfl_xor_sync(0xFFFFFFFFu, rs, o);
    if (lane == 0) rowsum[k] = rs;
    if (!v) return;
    constexpr int BCH = 8;
    for (int64_t b0 = 0; b0 < B; b0 += BCH) {
        float acc[BCH];
        float m[BCH];
#pragma unroll
        for (int q = 0; q < BCH; ++q) {
            acc[q] = 0.0f;
            m[q] = (b0 + q < B) ? mu[b0 + q] : 0.0f;
        }
        for (int64_t n = lane; n < N; n += 32) {
            const float wv = (float)code_value(w[n]);
#pragma unroll
            for (int q = 0; q < BCH; ++q)
                if (b0 + q < B) acc[q] = fmaf(colmean[(b0 + q) * N + n] - m[q], wv, acc[q]);
        }
#pragma unroll
        for (int q = 0; q < BCH; ++q) {
            float a = acc[q];
            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
            if (lane == 0 && b0 + q < B) v[(b0 + q) * K + k] = a;
        }
    }
}

// Two-way factors, first pass: per 128-row tile i and column k,
//   xs[i, k] = sum_{t in tile i} X8[t,k],   ps[i, k] = sum_{t in tile i} X8[t,k] eps[t].
template <typename CodeT>
__global__ void __launch_bounds__(128) ec_xsum_partial_kernel(const CodeT* X8, int64_t T, int64_t K,
                                                              const float* eps, int32_t* xs, float* ps) {
    const int64_t k = (int64_t)blockIdx.x * 128 + threadIdx.x;
    const int64_t i = blockIdx.y;
    if (k >= K) return;
    const int64_t t_end = min(T, (i + 1) * (int64_t)kTile);
    int32_t sx = 0;
    float sp = 0.0f;
    for (int64_t t = i * kTile; t < t_end; ++t) {
        const int x = code_value(X8[t * K + k]);
        sx += x;
        sp = fmaf((float)x, eps[t], sp);
    }
    xs[i * K + k] = sx;
    ps[i * K + k] = sp;
}

// Second pass: xsum[b, k] = sum over tiles of example b; p[k] = sum over all tiles.
__global__ void ec_xsum_reduce_kernel(const int32_t* xs, const float* ps, int64_t ntr, int64_t K, int64_t B,
                                      int64_t tiles_per_example, int32_t* xsum, float* p) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= K) return;
    float pk = 0.0f;
    for (int64_t b = 0; b < B; ++b) {
        const int64_t r0 = b * tiles_per_example, r1 = (B == 1) ? ntr : (b + 1) * tiles_per_example;
        int32_t s = 0;
        for (int64_t r = r0; r < r1; ++r) {
            s += xs[r * K + k];
            pk += ps[r * K + k];
        }
        xsum[b * K + k] = s;
    }
    p[k] = pk;
}

}  // namespace s3r

using namespace s3r;

extern "C" size_t s3r_ec_workspace_size(int64_t T, int64_t K) {
    if (T <= 0 || K <= 0) return 0;
    const size_t ntr = (size_t)s3r_cdiv(T, kTile);
    return ntr * (size_t)K * (sizeof(int32_t) + sizeof(float)) + 256;
}

extern "C" int s3r_ec_correct(const float* tok_err_part, const float* col_err_part, int64_t T, int64_t N, int64_t S,
                              const void* W8, int64_t K, const void* X8, int code_format, int ec_mode, float* eps,
                              float* mu, float* colmean, int32_t* rowsum, float* v, int32_t* xsum, float* p,
                              void* workspace, size_t workspace_bytes, int* d_status, cudaStream_t stream) {
    (void)d_status;
    if (T < 0 || N < 0 || K < 0 || S <= 0) return S3R_ERR_ARG;
    if (code_format != S3R_CODES_S8 && code_format != S3R_CODES_F16) return S3R_ERR_ARG;
    const bool f16 = code_format == S3R_CODES_F16;
    if (ec_mode != S3R_EC_NONE && ec_mode != S3R_EC_DX_ONLY && ec_mode != S3R_EC_TWO_WAY) return S3R_ERR_ARG;
    if (T == 0 || N == 0) return S3R_OK;
    if (T % S != 0) return S3R_ERR_SHAPE;
    if (S % kTile != 0 && S != T) return S3R_ERR_SHAPE;
    if (!tok_err_part || !col_err_part || !eps || !mu || !colmean) return S3R_ERR_ARG;
    const int64_t B = T / S, ntc = s3r_cdiv(N, kTile), ntr = s3r_cdiv(T, kTile);
    {
        const int64_t total = T + B * N;
        ec_means_kernel<<<(unsigned)s3r_cdiv(total, 256), 256, 0, stream>>>(tok_err_part, col_err_part, T, N, S, ntc,
                                                                          ntr, eps, colmean);
        S3R_CHECK_LAUNCH();
        ec_mu_kernel<<<(unsigned)B, 256, 0, stream>>>(eps, S, mu);
        S3R_CHECK_LAUNCH();
    }
    if (ec_mode == S3R_EC_NONE || K == 0) return S3R_OK;
    if (!W8 || !rowsum || !v) return S3R_ERR_ARG;
    if (f16)
        ec_gemv_kernel<<<(unsigned)s3r_cdiv(K, 8), 256, 0, stream>>>(static_cast<const __half*>(W8), K, N, B, colmean,
                                                                     mu, rowsum, v);
    else
        ec_gemv_kernel<<<(unsigned)s3r_cdiv(K, 8), 256, 0, stream>>>(static_cast<const int8_t*>(W8), K, N, B, colmean,
                                                                     mu, rowsum, v);
    S3R_CHECK_LAUNCH();
    if (ec_mode != S3R_EC_TWO_WAY) return S3R_OK;
    if (!X8 || !xsum || !p) return S3R_ERR_ARG;
    if (!workspace || workspace_bytes < s3r_ec_workspace_size(T, K)) return S3R_ERR_WORKSPACE;
    int32_t* xs = static_cast<int32_t*>(workspace);
    float* ps = reinterpret_cast<float*>(xs + ntr * K);
    dim3 grid((unsigned)s3r_cdiv(K, 128), (unsigned)ntr);
    if (f16)
        ec_xsum_partial_kernel<<<grid, 128, 0, stream>>>(static_cast<const __half*>(X8), T, K, eps, xs, ps);
    else
        ec_xsum_partial_kernel<<<grid, 128, 0, stream>>>(static_cast<const int8_t*>(X8), T, K, eps, xs, ps);
    S3R_CHECK_LAUNCH();
    ec_xsum_reduce_kernel<<<(unsigned)s3r_cdiv(K, 256), 256, 0, stream>>>(xs, ps, ntr, K, B, S / kTile, xsum, p);
    S3R_CHECK_LAUNCH();
    return S3R_OK;
}
