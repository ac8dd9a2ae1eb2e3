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

#include <cstdio>

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

// Generic (any row length) versions, one warp per weight row / one thread per
// column: used when rows are not a multiple of 8 codes.
template <typename CodeT>
__global__ void __launch_bounds__(256) ec_gemv_generic_kernel(const CodeT* W8, int64_t K, int64_t N, int64_t B,
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
    for (int64_t b = 0; b < B; ++b) {
        float a = 0.0f;
        const float m = mu[b];
        for (int64_t n = lane; n < N; n += 32) a = fmaf(colmean[b * N + n] - m, (float)code_value(w[n]), a);
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
        if (lane == 0) v[b * K + k] = a;
    }
}

template <typename CodeT>
__global__ void __launch_bounds__(128) ec_xsum_partial_generic_kernel(const CodeT* X8, int64_t T, int64_t K,
                                                                      const float* eps, int32_t* xs, float* ps,
                                                                      int64_t chunk) {
    const int64_t k = (int64_t)blockIdx.x * 128 + threadIdx.x;
    const int64_t c = blockIdx.y;
    if (k >= K) return;
    const int64_t t_end = min(T, (c + 1) * chunk);
    int32_t sx = 0;
    float sp = 0.0f;
    for (int64_t t = c * chunk; t < t_end; ++t) {
        const int x = code_value(X8[t * K + k]);
        sx += x;
        sp = fmaf((float)x, eps[t], sp);
    }
    xs[c * K + k] = sx;
    ps[c * K + k] = sp;
}

// 8 consecutive codes starting at p (16-byte aligned rows, 8-code chunks).
__device__ __forceinline__ void load8(const int8_t* p, float (&f)[8], int& isum) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    isum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int c = (int)(int8_t)(((i < 4 ? w.x : w.y) >> (8 * (i & 3))) & 0xFF);
        f[i] = (float)c;
        isum += c;
    }
}
__device__ __forceinline__ void load8(const __half* p, float (&f)[8], int& isum) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
    isum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        f[i] = __half2float(__ushort_as_half((unsigned short)(u[i >> 1] >> (16 * (i & 1)))));
        isum += (int)f[i];
    }
}

// rowsum[k] = sum_n W8[k,n] and v[b,k] = sum_n (colmean[b,n] - mu[b]) W8[k,n].
// One CTA per 8 weight rows; its 8 warps split the N range, each lane takes 8
// consecutive channels at a time (one 16-byte load per row), so the centered
// channel means are read once per CTA and reused for 8 rows.  Partial sums
// meet in shared memory in a fixed order.  Needs N % 8 == 0 and 16-byte rows;
// bmax examples per pass.
template <typename CodeT>
__global__ void __launch_bounds__(256) ec_gemv_kernel(const CodeT* W8, int64_t K, int64_t N, int64_t B,
                                                      const float* colmean, const float* mu, int32_t* rowsum,
                                                      float* v) {
    constexpr int ROWS = 8, BCH = 4;
    __shared__ float red_v[8][ROWS][BCH];
    __shared__ int red_r[8][ROWS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t k0 = (int64_t)blockIdx.x * ROWS;
    const int64_t nchunks = N / 8;                         // 8-channel chunks
    const int64_t per_warp = (nchunks + 7) / 8;
    const int64_t ch0 = warp * per_warp, ch1 = min(nchunks, ch0 + per_warp);
    for (int64_t b0 = 0; b0 < (B > 0 ? B : 1); b0 += BCH) {
        float acc[ROWS][BCH];
        int rs[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            rs[r] = 0;
#pragma unroll
            for (int q = 0; q < BCH; ++q) acc[r][q] = 0.0f;
        }
        float m[BCH];
#pragma unroll
        for (int q = 0; q < BCH; ++q) m[q] = (v && b0 + q < B) ? mu[b0 + q] : 0.0f;
        for (int64_t ch = ch0 + lane; ch < ch1; ch += 32) {
            const int64_t n = ch * 8;
            float cm[BCH][8];
#pragma unroll
            for (int q = 0; q < BCH; ++q) {
                if (v && b0 + q < B) {
                    const float4 x0 = __ldg(reinterpret_cast<const float4*>(colmean + (b0 + q) * N + n));
                    const float4 x1 = __ldg(reinterpret_cast<const float4*>(colmean + (b0 + q) * N + n + 4));
                    cm[q][0] = x0.x - m[q]; cm[q][1] = x0.y - m[q]; cm[q][2] = x0.z - m[q]; cm[q][3] = x0.w - m[q];
                    cm[q][4] = x1.x - m[q]; cm[q][5] = x1.y - m[q]; cm[q][6] = x1.z - m[q]; cm[q][7] = x1.w - m[q];
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) cm[q][i] = 0.0f;
                }
            }
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                if (k0 + r >= K) continue;
                float w[8];
                int isum;
                load8(W8 + (k0 + r) * N + n, w, isum);
                rs[r] += isum;
#pragma unroll
                for (int q = 0; q < BCH; ++q)
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[r][q] = fmaf(cm[q][i], w[i], acc[r][q]);
            }
        }
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) rs[r] += __shfl_xor_sync(0xFFFFFFFFu, rs[r], o);
#pragma unroll
            for (int q = 0; q < BCH; ++q)
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc[r][q] += __shfl_xor_sync(0xFFFFFFFFu, acc[r][q], o);
        }
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                red_r[warp][r] = rs[r];
#pragma unroll
                for (int q = 0; q < BCH; ++q) red_v[warp][r][q] = acc[r][q];
            }
        }
        __syncthreads();
        if (threadIdx.x < ROWS * BCH) {
            const int r = threadIdx.x / BCH, q = threadIdx.x % BCH;
            float sv = 0.0f;
            int sr = 0;
            for (int w = 0; w < 8; ++w) {
                sv += red_v[w][r][q];
                sr += red_r[w][r];
            }
            if (k0 + r < K) {
                if (b0 == 0 && q == 0) rowsum[k0 + r] = sr;
                if (v && b0 + q < B) v[(b0 + q) * K + k0 + r] = sv;
            }
        }
        __syncthreads();
        if (!v) break;
    }
}

// Two-way factors, first pass over row chunks of CH rows (each inside one
// example): per chunk c and column k, xs[c, k] = sum_t X8[t,k] and
// ps[c, k] = sum_t X8[t,k] eps[t].  A CTA covers 256 columns (8 per lane, one
// 16-byte load per row) and its 8 warps take every 8th row of the chunk.
constexpr int kXsumChunk = 128;
template <typename CodeT>
__global__ void __launch_bounds__(256) ec_xsum_partial_kernel(const CodeT* X8, int64_t T, int64_t K,
                                                              const float* eps, int32_t* xs, float* ps) {
    __shared__ float red_p[8][256];
    __shared__ int red_x[8][256];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t kc = (int64_t)blockIdx.x * 256 + 8 * lane;
    const int64_t c = blockIdx.y;
    const int64_t t0 = c * kXsumChunk, t1 = min(T, t0 + kXsumChunk);
    float sp[8];
    int sx[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) { sp[i] = 0.0f; sx[i] = 0; }
    if (kc < K) {
        for (int64_t t = t0 + warp; t < t1; t += 8) {
            float x[8];
            int isum;
            load8(X8 + t * K + kc, x, isum);
            const float e = __ldg(eps + t);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                sx[i] += (int)x[i];
                sp[i] = fmaf(x[i], e, sp[i]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        red_p[warp][8 * lane + i] = sp[i];
        red_x[warp][8 * lane + i] = sx[i];
    }
    __syncthreads();
    const int64_t k = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (k < K) {
        float a = 0.0f;
        int b = 0;
        for (int w = 0; w < 8; ++w) {
            a += red_p[w][threadIdx.x];
            b += red_x[w][threadIdx.x];
        }
        xs[c * K + k] = b;
        ps[c * K + k] = a;
    }
}

// Second pass: xsum[b, k] = sum over the chunks of example b; p[k] = sum over all chunks.
__global__ void ec_xsum_reduce_kernel(const int32_t* xs, const float* ps, int64_t nch, int64_t K, int64_t B,
                                      int64_t chunks_per_example, int32_t* xsum, float* p) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= K) return;
    float pk = 0.0f;
    for (int64_t b = 0; b < B; ++b) {
        const int64_t r0 = b * chunks_per_example, r1 = (B == 1) ? nch : (b + 1) * chunks_per_example;
        int32_t s = 0;
#pragma unroll 8
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
    const size_t nch = (size_t)s3r_cdiv(T, kXsumChunk);
    return nch * (size_t)K * (sizeof(int32_t) + sizeof(float)) + 256;
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
    // vector path: 8 codes per load, so rows (and colmean rows) must start on 16 bytes
    const bool vec_w = N % 8 == 0 && s3r_aligned16(W8) && s3r_aligned16(colmean);
    const unsigned gk = (unsigned)s3r_cdiv(K, 8);
    if (f16) {
        const __half* w = static_cast<const __half*>(W8);
        if (vec_w) ec_gemv_kernel<<<gk, 256, 0, stream>>>(w, K, N, B, colmean, mu, rowsum, v);
        else ec_gemv_generic_kernel<<<gk, 256, 0, stream>>>(w, K, N, B, colmean, mu, rowsum, v);
    } else {
        const int8_t* w = static_cast<const int8_t*>(W8);
        if (vec_w) ec_gemv_kernel<<<gk, 256, 0, stream>>>(w, K, N, B, colmean, mu, rowsum, v);
        else ec_gemv_generic_kernel<<<gk, 256, 0, stream>>>(w, K, N, B, colmean, mu, rowsum, v);
    }
    S3R_CHECK_LAUNCH();
    if (ec_mode != S3R_EC_TWO_WAY) return S3R_OK;
    if (!X8 || !xsum || !p) return S3R_ERR_ARG;
    if (!workspace || workspace_bytes < s3r_ec_workspace_size(T, K)) return S3R_ERR_WORKSPACE;
    const bool vec_x = K % 8 == 0 && s3r_aligned16(X8);
    const int64_t nch = s3r_cdiv(T, kXsumChunk);
    int32_t* xs = static_cast<int32_t*>(workspace);
    float* ps = reinterpret_cast<float*>(xs + nch * K);
    if (vec_x) {
        dim3 grid((unsigned)s3r_cdiv(K, 256), (unsigned)nch);
        if (f16) ec_xsum_partial_kernel<<<grid, 256, 0, stream>>>(static_cast<const __half*>(X8), T, K, eps, xs, ps);
        else ec_xsum_partial_kernel<<<grid, 256, 0, stream>>>(static_cast<const int8_t*>(X8), T, K, eps, xs, ps);
    } else {
        dim3 grid((unsigned)s3r_cdiv(K, 128), (unsigned)nch);
        if (f16)
            ec_xsum_partial_generic_kernel<<<grid, 128, 0, stream>>>(static_cast<const __half*>(X8), T, K, eps, xs, ps,
                                                                    kXsumChunk);
        else
            ec_xsum_partial_generic_kernel<<<grid, 128, 0, stream>>>(static_cast<const int8_t*>(X8), T, K, eps, xs, ps,
                                                                    kXsumChunk);
    }
    S3R_CHECK_LAUNCH();
    ec_xsum_reduce_kernel<<<(unsigned)s3r_cdiv(K, 256), 256, 0, stream>>>(xs, ps, nch, K, B, S / kXsumChunk, xsum,
                                                                          p);
    S3R_CHECK_LAUNCH();
    return S3R_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of s3r_ec_correct.
//
// Some callers cannot allocate device memory at the moment they run the
// backward: code that must not call cudaMalloc while a stream is being
// captured, code running from a host callback or a real-time loop where an
// allocation would block or fail, or deployments that fix their whole device
// memory budget before the first step.  For them the two-way column sums use a
// scratch array that lives in this library's module, not a caller workspace.
//
// The array is a file-scope __device__ object of kStaticScratchBytes (8 MiB):
// every GPU that loads the library holds it until the process exits.  Its
// name in host code is only a host-side stand-in, so the device address is
// fetched with cudaGetSymbolAddress, once per device, with that device
// current; the first call on a device does this set-up (call it once before
// any stream capture).  All calls share the array and it keeps the last
// call's contents; nothing in it needs to start at zero (every partial it
// holds is written before it is read).  Calls that overlap on the GPU (two
// streams, or two host threads) race on it.
// ---------------------------------------------------------------------------
#include <mutex>

namespace {
constexpr size_t kStaticScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_ec_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_ec_scratch on the current device (nullptr on failure).
void* static_scratch(int* status) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        *status = s3r_cuda_fail("s3r_ec_correct_static: cudaGetDevice", e == cudaSuccess ? cudaErrorInvalidDevice : e);
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_ec_scratch);
        if (e != cudaSuccess || !p) {
            (void)cudaGetLastError();
            *status = s3r_cuda_fail("s3r_ec_correct_static: cudaGetSymbolAddress", e == cudaSuccess ? cudaErrorUnknown : e);
            return nullptr;
        }
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}
}  // namespace

extern "C" int s3r_ec_correct_static(const float* tok_err_part, const float* col_err_part, int64_t T, int64_t N,
                                     int64_t S, const void* W8, int64_t K, const void* X8, int code_format,
                                     int ec_mode, float* eps, float* mu, float* colmean, int32_t* rowsum, float* v,
                                     int32_t* xsum, float* p, int* d_status, cudaStream_t stream) {
    if (ec_mode != S3R_EC_TWO_WAY)   // only the two-way factors need scratch
        return s3r_ec_correct(tok_err_part, col_err_part, T, N, S, W8, K, X8, code_format, ec_mode, eps, mu, colmean,
                              rowsum, v, xsum, p, nullptr, 0, d_status, stream);
    const size_t need = s3r_ec_workspace_size(T, K);
    if (need > kStaticScratchBytes) {
        char buf[200];
        std::snprintf(buf, sizeof(buf), "needs %zu bytes of scratch for T=%lld, K=%lld; the static array holds %zu",
                      need, (long long)T, (long long)K, kStaticScratchBytes);
        s3r_record_error("s3r_ec_correct_static", buf);
        return S3R_ERR_UNSUPPORTED;
    }
    int st = S3R_OK;
    void* scratch = static_scratch(&st);
    if (!scratch) return st;
    return s3r_ec_correct(tok_err_part, col_err_part, T, N, S, W8, K, X8, code_format, ec_mode, eps, mu, colmean,
                          rowsum, v, xsum, p, scratch, kStaticScratchBytes, d_status, stream);
}
