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
// deterministic run to run.  Up to two linears that share the input X (W1
// and W3 of the SwiGLU block) are handled by the same launches: their weight
// rows share one grid and the column sums of X are read once for both.
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>

#include "common.cuh"

namespace s3r {

__device__ __forceinline__ uint64_t ec_gtime() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ int code_value(int8_t c) { return c; }
__device__ __forceinline__ int code_value(__half c) { return __half2int_rn(c); }

constexpr int kMaxJobs = 2;

// One linear's statistics and factors (device pointers).
struct EcJob {
    const float* tok;      // [T, ntc] token error partials
    const float* col;      // [ntr, N] channel error partials
    const void* W8;        // [K, N] weight codes
    float* eps;            // [T]
    float* mu;             // [B]
    float* colmean;        // [B, N]
    int32_t* rowsum;       // [K]
    float* v;              // [B, K]
    int32_t* xsum;         // [B, K]
    float* p;              // [K]
};

struct EcMeansArgs {
    const float* tok[kMaxJobs];
    const float* col[kMaxJobs];
    float* eps[kMaxJobs];
    float* colmean[kMaxJobs];
    int64_t T, N, S, ntc, ntr;
    int* counter;          // column-block counters of the column-sum pass, zeroed here (or null)
    int ncounter;
};

// eps[t] = (sum_j tok[t, j]) / N ;  colmean[b, n] = (sum_{tile rows i of b} col[i, n]) / S
// (blockIdx.y selects the linear).
__global__ void ec_means_kernel(EcMeansArgs A) {
    const int j = blockIdx.y;
    const float* tok = j ? A.tok[1] : A.tok[0];
    const float* col = j ? A.col[1] : A.col[0];
    float* eps = j ? A.eps[1] : A.eps[0];
    float* colmean = j ? A.colmean[1] : A.colmean[0];
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t T = A.T, N = A.N, S = A.S, B = T / S;
    if (A.counter && blockIdx.x == 0 && j == 0)
        for (int c = threadIdx.x; c < A.ncounter; c += blockDim.x) A.counter[c] = 0;
    if (i < T) {
        float s = 0.0f;
        for (int64_t c = 0; c < A.ntc; ++c) s += tok[i * A.ntc + c];
        eps[i] = s / (float)N;
    } else if (i < T + B * N) {
        const int64_t k = i - T, b = k / N, n = k % N;
        int64_t r_begin, r_end;
        if (B == 1) { r_begin = 0; r_end = A.ntr; }
        else { r_begin = b * (S / kTile); r_end = (b + 1) * (S / kTile); }
        float s = 0.0f;
        for (int64_t r = r_begin; r < r_end; ++r) s += col[r * N + n];
        colmean[b * N + n] = s / (float)S;
    }
}

// mu[b] = (sum_{t < S} e[b S + t]) / S for b0 <= b < b0 + 8 (and b < B) over a
// CTA of NT threads in a fixed order: per-thread strided sums, then a tree
// over the NT partials.  The loads of all eight examples are in flight
// together.  red holds 8 x NT floats; the results land in out[b].  Every
// caller with the same NT gets the same bits.
template <int NT>
__device__ void cta_means8(const float* e, int64_t S, int64_t B, int64_t b0, float* red, float* out) {
    float s[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) s[q] = 0.0f;
#pragma unroll 4
    for (int64_t t = threadIdx.x; t < S; t += NT) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (b0 + q < B) s[q] += e[(b0 + q) * S + t];
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) red[q * NT + threadIdx.x] = s[q];
    __syncthreads();
    for (int w = NT / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w)
#pragma unroll
            for (int q = 0; q < 8; ++q) red[q * NT + threadIdx.x] += red[q * NT + threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x < 8 && b0 + threadIdx.x < B) out[b0 + threadIdx.x] = red[threadIdx.x * NT] / (float)S;
    __syncthreads();
}

constexpr int kGemvThreads = 512;

// mu[b] = (1/S) sum_{t in b} eps[t]  (used where the factor kernels do not run)
__global__ void __launch_bounds__(kGemvThreads) ec_mu_kernel(const float* eps, int64_t S, int64_t B, float* mu) {
    __shared__ float red[8 * kGemvThreads];
    cta_means8<kGemvThreads>(eps, S, B, (int64_t)blockIdx.x * 8, red, mu);
}

// ---------------------------------------------------------------------------
// Generic (any row length) versions, one warp per weight row / one thread per
// column: used when rows are not a multiple of 8 codes or not 16-byte aligned.
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

constexpr int kXsumChunk = 128;   // rows per column-sum chunk (inside one example)

template <typename CodeT>
__global__ void __launch_bounds__(128) ec_xsum_partial_generic_kernel(const CodeT* X8, int64_t T, int64_t K,
                                                                      const float* eps, int32_t* xs, float* ps) {
    const int64_t k = (int64_t)blockIdx.x * 128 + threadIdx.x;
    const int64_t c = blockIdx.y;
    if (k >= K) return;
    const int64_t t_end = min(T, (c + 1) * kXsumChunk);
    int32_t sx = 0;
    float sp = 0.0f;
    for (int64_t t = c * kXsumChunk; t < t_end; ++t) {
        const int x = code_value(X8[t * K + k]);
        sx += x;
        sp = fmaf((float)x, eps[t], sp);
    }
    xs[c * K + k] = sx;
    ps[c * K + k] = sp;
}

// xsum[b, k] = sum over the chunks of example b; p[k] = sum over all chunks.
__global__ void ec_xsum_reduce_generic_kernel(const int32_t* xs, const float* ps, int64_t nch, int64_t K, int64_t B,
                                              int64_t chunks_per_example, int32_t* xsum, float* p) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= K) return;
    float pk = 0.0f;
    for (int64_t b = 0; b < B; ++b) {
        const int64_t r0 = b * chunks_per_example, r1 = (B == 1) ? nch : (b + 1) * chunks_per_example;
        int32_t s = 0;
        for (int64_t r = r0; r < r1; ++r) {
            s += xs[r * K + k];
            pk += ps[r * K + k];
        }
        xsum[b * K + k] = s;
    }
    p[k] = pk;
}

// ---------------------------------------------------------------------------
// Vector path (rows of 8-code multiples, 16-byte aligned).

// rowsum[k] = sum_n W8[k,n] and v[b,k] = sum_n (colmean[b,n] - mu[b]) W8[k,n].
// One 512-thread CTA per SM.  Each CTA first computes every mu[b] (fixed
// order, the same bits in every CTA; the first CTA of a linear stores them).
// A warp owns up to kGemvPairs pairs of weight rows (pairs strided over all
// warps of the linear) and keeps their sums in registers while the CTA walks
// the examples kGemvBch at a time and the channels in slabs of `slab`: the
// centered means of a slab are staged in shared memory, and the lanes stride
// each row 8 codes (one 16-byte load) at a time with the loads of
// kGemvUnroll chunks in flight.  The row sums meet in a butterfly after the
// last slab.  CTAs [0, ctas0) serve linear 0, the rest linear 1.
constexpr int kGemvRows = 2, kGemvBch = 4, kGemvUnroll = 8, kGemvPairs = 3;
constexpr int kGemvWarps = kGemvThreads / 32;
constexpr int64_t kGemvSlabFloats = 24 * 1024;   // staged means per slab (all kGemvBch examples): 96 KiB

struct EcGemvArgs {
    const void* W8[kMaxJobs];
    const float* colmean[kMaxJobs];
    const float* eps[kMaxJobs];
    float* mu[kMaxJobs];
    int32_t* rowsum[kMaxJobs];
    float* v[kMaxJobs];
    int64_t K, N, S, B;
    int64_t slab;                // channels per staged slab (multiple of 8)
    int ctas0, ctas1;
};

// dynamic shared memory: 8 x 512 floats (reductions) + B rounded to 4 + kGemvBch * slab
static size_t gemv_smem_bytes(int64_t slab, int64_t B) {
    return (size_t)(8 * kGemvThreads + ((B + 3) & ~(int64_t)3) + kGemvBch * slab) * sizeof(float);
}

template <typename CodeT>
__device__ __forceinline__ uint4 raw8(const CodeT* p) {
    if (sizeof(CodeT) == 2) return __ldg(reinterpret_cast<const uint4*>(p));
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
    return make_uint4(w.x, w.y, 0u, 0u);
}
// the 8 codes of a raw 16-byte (fp16) or 8-byte (int8) load as floats
__device__ __forceinline__ void codes8(const uint4& w, float (&f)[8], __half) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = __half2float(__ushort_as_half((unsigned short)(u[i >> 1] >> (16 * (i & 1)))));
}
__device__ __forceinline__ void codes8(const uint4& w, float (&f)[8], int8_t) {
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = (float)(int)(int8_t)(((i < 4 ? w.x : w.y) >> (8 * (i & 3))) & 0xFF);
}

template <typename CodeT>
__global__ void __launch_bounds__(kGemvThreads) ec_gemv_kernel(EcGemvArgs A) {
    extern __shared__ __align__(16) float sm[];
    const int64_t K = A.K, N = A.N, S = A.S, B = A.B, slab = A.slab;
    float* red = sm;
    float* mu_s = sm + 8 * kGemvThreads;
    float* cm = mu_s + ((B + 3) & ~(int64_t)3);   // [kGemvBch][slab]
    const int j = (int)blockIdx.x < A.ctas0 ? 0 : 1;
    const CodeT* W8 = static_cast<const CodeT*>(j ? A.W8[1] : A.W8[0]);
    const float* colmean = j ? A.colmean[1] : A.colmean[0];
    const float* eps = j ? A.eps[1] : A.eps[0];
    int32_t* rowsum = j ? A.rowsum[1] : A.rowsum[0];
    float* v = j ? A.v[1] : A.v[0];
    const int64_t cta = j ? blockIdx.x - A.ctas0 : blockIdx.x;
    const int64_t nctas = j ? A.ctas1 : A.ctas0;
    for (int64_t b0 = 0; b0 < B; b0 += 8) cta_means8<kGemvThreads>(eps, S, B, b0, red, mu_s);
    if (cta == 0) {
        float* mu = j ? A.mu[1] : A.mu[0];
        for (int64_t b = threadIdx.x; b < B; b += kGemvThreads) mu[b] = mu_s[b];
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t gw = cta * kGemvWarps + warp, nw = nctas * kGemvWarps;
    for (int64_t b0 = 0; b0 < B; b0 += kGemvBch) {
        float acc[kGemvPairs][kGemvRows][kGemvBch];
        int rs[kGemvPairs][kGemvRows];
#pragma unroll
        for (int pp = 0; pp < kGemvPairs; ++pp)
#pragma unroll
            for (int r = 0; r < kGemvRows; ++r) {
                rs[pp][r] = 0;
#pragma unroll
                for (int q = 0; q < kGemvBch; ++q) acc[pp][r][q] = 0.0f;
            }
        for (int64_t n0 = 0; n0 < N; n0 += slab) {
            const int64_t ns = N - n0 < slab ? N - n0 : slab;   // channels in this slab (multiple of 8)
            __syncthreads();   // the previous slab is done with cm
#pragma unroll
            for (int q = 0; q < kGemvBch; ++q) {
                const bool on = b0 + q < B;
                const float m = on ? mu_s[b0 + q] : 0.0f;
                for (int64_t i = threadIdx.x; i < ns / 4; i += kGemvThreads) {
                    float4 c = on ? __ldg(reinterpret_cast<const float4*>(colmean + (b0 + q) * N + n0) + i)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
                    c.x -= m; c.y -= m; c.z -= m; c.w -= m;
                    reinterpret_cast<float4*>(cm + q * slab)[i] = on ? c : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            __syncthreads();
            const int64_t nch = ns / 8;
#pragma unroll
            for (int pp = 0; pp < kGemvPairs; ++pp) {
                const int64_t k0 = (gw + pp * nw) * kGemvRows;
                if (k0 >= K) break;
                const CodeT* wrow[kGemvRows];
#pragma unroll
                for (int r = 0; r < kGemvRows; ++r) wrow[r] = W8 + (k0 + r < K ? k0 + r : K - 1) * N + n0;   // clamped
                for (int64_t c0 = 0; c0 < nch; c0 += 32 * kGemvUnroll) {
                    uint4 raw[kGemvUnroll][kGemvRows];
#pragma unroll
                    for (int u = 0; u < kGemvUnroll; ++u) {
                        const int64_t ch = c0 + 32 * u + lane;
                        const int64_t chc = ch < nch ? ch : nch - 1;   // clamped: always a valid load
#pragma unroll
                        for (int r = 0; r < kGemvRows; ++r) raw[u][r] = raw8(wrow[r] + 8 * chc);
                    }
#pragma unroll
                    for (int u = 0; u < kGemvUnroll; ++u) {
                        const int64_t ch = c0 + 32 * u + lane;
                        if (ch >= nch) break;
                        float w[kGemvRows][8];
#pragma unroll
                        for (int r = 0; r < kGemvRows; ++r) {
                            codes8(raw[u][r], w[r], CodeT{});
#pragma unroll
                            for (int i = 0; i < 8; ++i) rs[pp][r] += (int)w[r][i];
                        }
#pragma unroll
                        for (int q = 0; q < kGemvBch; ++q) {
                            const float4 x0 = *reinterpret_cast<const float4*>(cm + q * slab + 8 * ch);
                            const float4 x1 = *reinterpret_cast<const float4*>(cm + q * slab + 8 * ch + 4);
                            const float c[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                            for (int r = 0; r < kGemvRows; ++r)
#pragma unroll
                                for (int i = 0; i < 8; ++i) acc[pp][r][q] = fmaf(c[i], w[r][i], acc[pp][r][q]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int pp = 0; pp < kGemvPairs; ++pp) {
            const int64_t k0 = (gw + pp * nw) * kGemvRows;
            if (k0 >= K) break;
#pragma unroll
            for (int r = 0; r < kGemvRows; ++r) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) rs[pp][r] += __shfl_xor_sync(0xFFFFFFFFu, rs[pp][r], o);
#pragma unroll
                for (int q = 0; q < kGemvBch; ++q)
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) acc[pp][r][q] += __shfl_xor_sync(0xFFFFFFFFu, acc[pp][r][q], o);
            }
            if (lane == 0) {
#pragma unroll
                for (int r = 0; r < kGemvRows; ++r) {
                    if (k0 + r >= K) continue;
                    if (b0 == 0) rowsum[k0 + r] = rs[pp][r];
#pragma unroll
                    for (int q = 0; q < kGemvBch; ++q)
                        if (b0 + q < B) v[(b0 + q) * K + k0 + r] = acc[pp][r][q];
                }
            }
        }
    }
}

// Two-way factors over X8 [T, K]: xsum[b, k] = sum_{t in b} X8[t,k] and, per
// linear j, p_j[k] = sum_t X8[t,k] eps_j[t].  CTA (cb, c) sums the
// ROWS-row chunk c over 256 columns (8 per lane, one 16-byte load per
// row; warp w takes rows w, w + 8, ..., all of its loads in flight together)
// into workspace partials; the last CTA of each column block (a counter, no
// waiting) adds the chunks up in a fixed order, one column per thread.
constexpr int kXsumGroup = 16;   // rows whose loads are issued together

struct EcXsumArgs {
    const void* X8;
    int64_t T, K, S, B;
    const float* eps[kMaxJobs];
    int32_t* xsum[kMaxJobs];   // xsum is the same for every linear; each gets its copy
    float* p[kMaxJobs];
    int32_t* xs;               // [nch, K]
    float* ps;                 // [NJ, nch, K]
    int* counter;              // [K / 256]
};

template <typename CodeT, int NJ, int ROWS>
__global__ void __launch_bounds__(256) ec_xsum_kernel(EcXsumArgs A) {
    constexpr int kXsumRowsPerWarp = ROWS / 8;
    constexpr int P = 33;   // padded pitch: conflict-free writes (lane-major) and reads (column-major)
    __shared__ float red_p[NJ][8][8 * P];
    __shared__ int red_x[8][8 * P];
    __shared__ int last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t T = A.T, K = A.K;
    const int64_t nch = gridDim.y, c = blockIdx.y;
    const int64_t kc = (int64_t)blockIdx.x * 256 + 8 * lane;
    const int64_t t0 = c * ROWS;
    const CodeT* X8 = static_cast<const CodeT*>(A.X8);
    const int64_t kcl = kc < K ? kc : K - 8;   // clamped column: always a valid load
    {
        float sp[NJ][8];
        int sx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            sx[i] = 0;
#pragma unroll
            for (int jj = 0; jj < NJ; ++jj) sp[jj][i] = 0.0f;
        }
#pragma unroll
        for (int g = 0; g < kXsumRowsPerWarp; g += kXsumGroup) {
            uint4 raw[kXsumGroup];
            float e[NJ][kXsumGroup];
#pragma unroll
            for (int u = 0; u < kXsumGroup; ++u) {
                const int64_t t = t0 + warp + 8 * (g + u);
                const int64_t tc = t < T ? t : T - 1;   // clamped row
                raw[u] = raw8(X8 + tc * K + kcl);
#pragma unroll
                for (int jj = 0; jj < NJ; ++jj) e[jj][u] = t < T ? __ldg(A.eps[jj] + tc) : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < kXsumGroup; ++u) {
                const int64_t t = t0 + warp + 8 * (g + u);
                float x[8];
                codes8(raw[u], x, CodeT{});
                if (t < T && kc < K) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) sx[i] += (int)x[i];
                }
#pragma unroll
                for (int jj = 0; jj < NJ; ++jj)
#pragma unroll
                    for (int i = 0; i < 8; ++i) sp[jj][i] = fmaf(x[i], e[jj][u], sp[jj][i]);
            }
        }
        // column 8 * lane + i of this block sits at [i * P + lane]
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            red_x[warp][i * P + lane] = sx[i];
#pragma unroll
            for (int jj = 0; jj < NJ; ++jj) red_p[jj][warp][i * P + lane] = sp[jj][i];
        }
    }
    __syncthreads();
    const int64_t k = (int64_t)blockIdx.x * 256 + threadIdx.x;
    const int slot = (threadIdx.x & 7) * P + (threadIdx.x >> 3);
    if (k < K) {
        int xb = 0;
        float a[NJ];
#pragma unroll
        for (int jj = 0; jj < NJ; ++jj) a[jj] = 0.0f;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            xb += red_x[w][slot];
#pragma unroll
            for (int jj = 0; jj < NJ; ++jj) a[jj] += red_p[jj][w][slot];
        }
        A.xs[c * K + k] = xb;
#pragma unroll
        for (int jj = 0; jj < NJ; ++jj) A.ps[(jj * nch + c) * K + k] = a[jj];
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(A.counter + blockIdx.x, 1) == (int)nch - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    // Last CTA of this column block: thread = column; per example the chunks
    // are added in order, then p adds the examples in order.
    if (k < K) {
        const int64_t B = A.B, cpe = B == 1 ? nch : A.S / ROWS;
        float pk[NJ];
#pragma unroll
        for (int jj = 0; jj < NJ; ++jj) pk[jj] = 0.0f;
        for (int64_t b = 0; b < B; ++b) {
            int xb = 0;
            float pb[NJ];
#pragma unroll
            for (int jj = 0; jj < NJ; ++jj) pb[jj] = 0.0f;
#pragma unroll 8
            for (int64_t cc = b * cpe; cc < (b + 1) * cpe; ++cc) {
                xb += __ldcg(A.xs + cc * K + k);
#pragma unroll
                for (int jj = 0; jj < NJ; ++jj) pb[jj] += __ldcg(A.ps + (jj * nch + cc) * K + k);
            }
#pragma unroll
            for (int jj = 0; jj < NJ; ++jj) {
                A.xsum[jj][b * K + k] = xb;
                pk[jj] += pb[jj];
            }
        }
#pragma unroll
        for (int jj = 0; jj < NJ; ++jj) A.p[jj][k] = pk[jj];
    }
    if (threadIdx.x == 0) A.counter[blockIdx.x] = 0;
}

// fp16 codes: the same sums streamed through shared memory.  One CTA per SM
// walks the (column block, row chunk) items; TMA copies 64-row x 256-column
// boxes (32 KiB) into a 4-stage ring while the warps accumulate the previous
// ones (warp w takes rows w, w + 8, ... of a box, lane l columns 8l .. 8l+7;
// the integer sums are exact in fp32: at most 256 * 127 per chunk).  Partials,
// counters and the final fixed-order reduction as in ec_xsum_kernel.
constexpr int kXsStages = 4, kXsBoxRows = 64;
constexpr int kXsBoxBytes = kXsBoxRows * 256 * 2;
constexpr int kXsSmem = kXsStages * kXsBoxBytes + 128 + 64;

__device__ __forceinline__ bool xs_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = ec_gtime();
    while (true) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
        if (ec_gtime() - t0 > 2000000000ull) return false;
    }
}

template <int NJ, int ROWS>
__global__ void __launch_bounds__(256, 1)
    ec_xsum_tma_kernel(const __grid_constant__ CUtensorMap tmX, EcXsumArgs A, int64_t ncb, int64_t nch,
                       int* d_status) {
    constexpr int P = 33;
    constexpr int NBOX = ROWS / kXsBoxRows;
    extern __shared__ uint8_t xsm_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(xsm_raw) + 127) & ~(uintptr_t)127);
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + kXsStages * kXsBoxBytes);
    __shared__ float red_p[NJ][8][8 * P];
    __shared__ float red_x[8][8 * P];
    __shared__ int last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t T = A.T, K = A.K;
    const int64_t nitems = ncb * nch;
    const int64_t my_items = (int64_t)blockIdx.x < nitems ? (nitems - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int64_t total = my_items * NBOX;   // boxes this CTA streams
    auto box_item = [&](int64_t kk) { return (int64_t)blockIdx.x + (kk / NBOX) * gridDim.x; };
    auto issue = [&](int64_t kk) {
        const int64_t item = box_item(kk);
        const int s = (int)(kk % kXsStages);
        const uint32_t bar = (uint32_t)__cvta_generic_to_shared(full + s);
        const int32_t x = (int32_t)((item % ncb) * 256), y = (int32_t)((item / ncb) * ROWS + (kk % NBOX) * kXsBoxRows);
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(kXsBoxBytes) : "memory");
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
            ::"r"((uint32_t)__cvta_generic_to_shared(ring + s * kXsBoxBytes)), "l"((uint64_t)&tmX), "r"(x), "r"(y),
            "r"(bar)
            : "memory");
    };
    if (threadIdx.x == 0) {
        for (int i = 0; i < kXsStages; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"((uint32_t)__cvta_generic_to_shared(full + i))
                         : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmX) : "memory");
    }
    __syncthreads();
    int64_t issued = 0;   // thread 0's count
    if (threadIdx.x == 0)
        for (; issued < kXsStages && issued < total; ++issued) issue(issued);
    int64_t kk = 0;
    bool ok = true;
    for (int64_t k = 0; k < my_items && ok; ++k) {
        const int64_t item = (int64_t)blockIdx.x + k * gridDim.x;
        const int64_t cb = item % ncb, c = item / ncb;
        float2 sx[4], sp[NJ][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            sx[i] = make_float2(0.f, 0.f);
#pragma unroll
            for (int jj = 0; jj < NJ; ++jj) sp[jj][i] = make_float2(0.f, 0.f);
        }
        for (int box = 0; box < NBOX; ++box, ++kk) {
            const int s = (int)(kk % kXsStages);
            // every thread waits; the CTA leaves together if any wait ran out
            if (!__syncthreads_and(xs_wait((uint32_t)__cvta_generic_to_shared(full + s),
                                           (uint32_t)((kk / kXsStages) & 1)))) {
                if (threadIdx.x == 0 && d_status) *(volatile int*)d_status = S3R_ERR_TIMEOUT;
                ok = false;
                break;
            }
            const uint8_t* st = ring + s * kXsBoxBytes;
            const int64_t tb = c * ROWS + box * kXsBoxRows;
#pragma unroll
            for (int i = 0; i < kXsBoxRows / 8; ++i) {
                const int r = warp + 8 * i;
                const int64_t t = tb + r;
                const uint4 w = *reinterpret_cast<const uint4*>(st + (r * 256 + 8 * lane) * 2);
                const uint32_t u[4] = {w.x, w.y, w.z, w.w};
                float e[NJ];
#pragma unroll
                for (int jj = 0; jj < NJ; ++jj) e[jj] = t < T ? __ldg(A.eps[jj] + t) : 0.0f;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&u[q]));
                    sx[q] = f2_add(sx[q], x);
#pragma unroll
                    for (int jj = 0; jj < NJ; ++jj) sp[jj][q] = f2_fma(x, make_float2(e[jj], e[jj]), sp[jj][q]);
                }
            }
            __syncthreads();   // every thread is done with this stage
            if (threadIdx.x == 0 && issued < total) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue(issued);
                ++issued;
            }
        }
        if (!ok) break;
        // the chunk's column sums: warps meet in shared memory in warp order
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            red_x[warp][(2 * q) * P + lane] = sx[q].x;
            red_x[warp][(2 * q + 1) * P + lane] = sx[q].y;
#pragma unroll
            for (int jj = 0; jj < NJ; ++jj) {
                red_p[jj][warp][(2 * q) * P + lane] = sp[jj][q].x;
                red_p[jj][warp][(2 * q + 1) * P + lane] = sp[jj][q].y;
            }
        }
        __syncthreads();
        const int64_t kcol = cb * 256 + threadIdx.x;
        const int slot = (threadIdx.x & 7) * P + (threadIdx.x >> 3);
        if (kcol < K) {
            float xb = 0.0f;
            float a[NJ];
#pragma unroll
            for (int jj = 0; jj < NJ; ++jj) a[jj] = 0.0f;
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                xb += red_x[w][slot];
#pragma unroll
                for (int jj = 0; jj < NJ; ++jj) a[jj] += red_p[jj][w][slot];
            }
            A.xs[c * K + kcol] = (int32_t)xb;
#pragma unroll
            for (int jj = 0; jj < NJ; ++jj) A.ps[(jj * nch + c) * K + kcol] = a[jj];
        }
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) last = atomicAdd(A.counter + cb, 1) == (int)nch - 1;
        __syncthreads();
        if (last && kcol < K) {
            __threadfence();
            // last chunk of this column block: thread = column, chunks in order per example
            const int64_t B = A.B, cpe = B == 1 ? nch : A.S / ROWS;
            float pk[NJ];
#pragma unroll
            for (int jj = 0; jj < NJ; ++jj) pk[jj] = 0.0f;
            for (int64_t b = 0; b < B; ++b) {
                int xbi = 0;
                float pb[NJ];
#pragma unroll
                for (int jj = 0; jj < NJ; ++jj) pb[jj] = 0.0f;
#pragma unroll 8
                for (int64_t cc = b * cpe; cc < (b + 1) * cpe; ++cc) {
                    xbi += __ldcg(A.xs + cc * K + kcol);
#pragma unroll
                    for (int jj = 0; jj < NJ; ++jj) pb[jj] += __ldcg(A.ps + (jj * nch + cc) * K + kcol);
                }
#pragma unroll
                for (int jj = 0; jj < NJ; ++jj) {
                    A.xsum[jj][b * K + kcol] = xbi;
                    pk[jj] += pb[jj];
                }
            }
#pragma unroll
            for (int jj = 0; jj < NJ; ++jj) A.p[jj][kcol] = pk[jj];
        }
        if (last && threadIdx.x == 0) A.counter[cb] = 0;
        __syncthreads();   // red_* and `last` are reused by the next item
    }
    // an early exit may leave copies in flight: wait for them before leaving
    if (threadIdx.x == 0)
        for (int64_t q = kk; q < issued; ++q)
            xs_wait((uint32_t)__cvta_generic_to_shared(full + (q % kXsStages)), (uint32_t)((q / kXsStages) & 1));
}

static PFN_cuTensorMapEncodeTiled_v12000 ec_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess && p)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            (void)cudaGetLastError();
    }
    return fn;
}

static int ec_sm_count() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            (void)cudaGetLastError();
            n = 148;
        }
    }
    return n;
}

template <int NJ, int ROWS>
static int launch_xsum_tma_t(const CUtensorMap& map, const EcXsumArgs& X, int64_t ncb, int64_t nch, int* d_status,
                             cudaStream_t stream) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e =
            cudaFuncSetAttribute(ec_xsum_tma_kernel<NJ, ROWS>, cudaFuncAttributeMaxDynamicSharedMemorySize, kXsSmem);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return s3r_cuda_fail("ec column sums: cudaFuncSetAttribute", e);
        }
        attr = true;
    }
    const int64_t items = ncb * nch;
    const int64_t grid = std::min<int64_t>(items, ec_sm_count());
    ec_xsum_tma_kernel<NJ, ROWS><<<(unsigned)grid, 256, kXsSmem, stream>>>(map, X, ncb, nch, d_status);
    S3R_CHECK_LAUNCH();
    return S3R_OK;
}

// fp16 codes X8 [T, K] with 16-byte aligned rows: the TMA column-sum kernel.
// Returns 1 when it does not apply (the caller falls back to ec_xsum_kernel).
static int launch_xsum_tma(const EcXsumArgs& X, int nj, bool wide, int64_t ncb, int64_t nch, int* d_status,
                           cudaStream_t stream) {
    auto fn = ec_encode_fn();
    if (!fn || X.T >= (int64_t(1) << 31) || X.K >= (int64_t(1) << 31)) return 1;
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)X.K, (cuuint64_t)X.T};
    const cuuint64_t strides[1] = {(cuuint64_t)X.K * 2};
    const cuuint32_t box[2] = {256, (cuuint32_t)kXsBoxRows};
    const cuuint32_t estr[2] = {1, 1};
    // rows and columns past the end read as zero
    CUresult r = fn(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(X.X8), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return 1;
    if (wide) return nj == 2 ? launch_xsum_tma_t<2, 256>(map, X, ncb, nch, d_status, stream)
                             : launch_xsum_tma_t<1, 256>(map, X, ncb, nch, d_status, stream);
    return nj == 2 ? launch_xsum_tma_t<2, 128>(map, X, ncb, nch, d_status, stream)
                   : launch_xsum_tma_t<1, 128>(map, X, ncb, nch, d_status, stream);
}

// Workspace of the column-sum pass for `njobs` linears sharing X8 [T, K].
static size_t xsum_workspace_bytes(int64_t T, int64_t K, int njobs) {
    const size_t nch = (size_t)s3r_cdiv(T, kXsumChunk);   // the generic path's chunks, the finer of the two
    return nch * (size_t)K * (sizeof(int32_t) + njobs * sizeof(float)) + (size_t)s3r_cdiv(K, 256) * sizeof(int) +
           512;
}

template <typename CodeT>
static int launch_factors(const EcJob* jobs, int nj, int64_t T, int64_t N, int64_t S, int64_t K, const void* X8,
                          int ec_mode, void* workspace, size_t workspace_bytes, int* d_status,
                          cudaStream_t stream) {
    const int64_t B = T / S, ntc = s3r_cdiv(N, kTile), ntr = s3r_cdiv(T, kTile);
    const bool two = ec_mode == S3R_EC_TWO_WAY;
    bool vec_w = N % 8 == 0;
    for (int j = 0; j < nj; ++j) vec_w = vec_w && s3r_aligned16(jobs[j].W8) && s3r_aligned16(jobs[j].colmean);
    const int64_t slab = std::min<int64_t>(N, kGemvSlabFloats / kGemvBch);   // multiple of 8 when N is
    const size_t gsm = gemv_smem_bytes(slab, B);
    vec_w = vec_w && gsm <= 200 * 1024;
    // every warp holds at most kGemvPairs row pairs: one CTA per SM gives sms * kGemvWarps warps per launch
    int gsms = 148;
    {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&gsms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            (void)cudaGetLastError();
            gsms = 148;
        }
    }
    const int64_t per_job = std::max<int64_t>(1, gsms / nj);
    vec_w = vec_w && s3r_cdiv(K, kGemvRows) <= per_job * kGemvWarps * kGemvPairs;
    const bool vec_x = K % 8 == 0 && s3r_aligned16(X8);
    // workspace: xs [nch, K] | ps [nj, nch, K] | counters
    const int64_t nch = s3r_cdiv(T, kXsumChunk), ncb = s3r_cdiv(K, 256);
    int32_t* xs = nullptr;
    float* ps = nullptr;
    int* counter = nullptr;
    if (two) {
        if (!workspace || workspace_bytes < xsum_workspace_bytes(T, K, nj)) return S3R_ERR_WORKSPACE;
        uintptr_t base = ((uintptr_t)workspace + 255) & ~(uintptr_t)255;
        xs = reinterpret_cast<int32_t*>(base);
        ps = reinterpret_cast<float*>(xs + nch * K);
        counter = reinterpret_cast<int*>(ps + nj * nch * K);
    }
    {
        EcMeansArgs M{};
        for (int j = 0; j < nj; ++j) {
            M.tok[j] = jobs[j].tok;
            M.col[j] = jobs[j].col;
            M.eps[j] = jobs[j].eps;
            M.colmean[j] = jobs[j].colmean;
        }
        M.T = T; M.N = N; M.S = S; M.ntc = ntc; M.ntr = ntr;
        M.counter = (two && vec_x) ? counter : nullptr;
        M.ncounter = (int)ncb;
        dim3 grid((unsigned)s3r_cdiv(T + B * N, 256), (unsigned)nj);
        ec_means_kernel<<<grid, 256, 0, stream>>>(M);
        S3R_CHECK_LAUNCH();
    }
    if (ec_mode == S3R_EC_NONE || K == 0 || !vec_w) {
        for (int j = 0; j < nj; ++j) {
            ec_mu_kernel<<<(unsigned)s3r_cdiv(B, 8), kGemvThreads, 0, stream>>>(jobs[j].eps, S, B, jobs[j].mu);
            S3R_CHECK_LAUNCH();
        }
    }
    if (ec_mode == S3R_EC_NONE || K == 0) return S3R_OK;
    if (vec_w) {
        EcGemvArgs G{};
        for (int j = 0; j < nj; ++j) {
            G.W8[j] = jobs[j].W8;
            G.colmean[j] = jobs[j].colmean;
            G.eps[j] = jobs[j].eps;
            G.mu[j] = jobs[j].mu;
            G.rowsum[j] = jobs[j].rowsum;
            G.v[j] = jobs[j].v;
        }
        G.K = K; G.N = N; G.S = S; G.B = B; G.slab = slab;
        // persistent: one CTA per SM in all, split evenly between the linears
        const int64_t need = s3r_cdiv(K, kGemvWarps * kGemvRows);   // CTAs that give every warp a row pair
        const int64_t per = std::min<int64_t>(need, per_job);
        G.ctas0 = (int)per;
        G.ctas1 = nj > 1 ? (int)per : 0;
        static bool attr = false;
        if (!attr) {
            cudaError_t e = cudaFuncSetAttribute(ec_gemv_kernel<CodeT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 200 * 1024);
            if (e != cudaSuccess) {
                (void)cudaGetLastError();
                return s3r_cuda_fail("ec gemv: cudaFuncSetAttribute", e);
            }
            attr = true;
        }
        ec_gemv_kernel<CodeT><<<(unsigned)(per * nj), kGemvThreads, gsm, stream>>>(G);
        S3R_CHECK_LAUNCH();
    } else {
        for (int j = 0; j < nj; ++j) {
            ec_gemv_generic_kernel<<<(unsigned)s3r_cdiv(K, 8), 256, 0, stream>>>(
                static_cast<const CodeT*>(jobs[j].W8), K, N, B, jobs[j].colmean, jobs[j].mu, jobs[j].rowsum,
                jobs[j].v);
            S3R_CHECK_LAUNCH();
        }
    }
    if (!two) return S3R_OK;
    if (vec_x) {
        EcXsumArgs X{};
        X.X8 = X8; X.T = T; X.K = K; X.S = S; X.B = B;
        for (int j = 0; j < nj; ++j) {
            X.eps[j] = jobs[j].eps;
            X.xsum[j] = jobs[j].xsum;
            X.p[j] = jobs[j].p;
        }
        X.xs = xs; X.ps = ps; X.counter = counter;
        // 256-row chunks where the examples allow it (chunks never straddle two)
        const bool wide = B == 1 || S % 256 == 0;
        const int64_t nchw = s3r_cdiv(T, wide ? 256 : 128);
        if (sizeof(CodeT) == 2) {
            int st = launch_xsum_tma(X, nj, wide, ncb, nchw, d_status, stream);
            if (st <= 0) return st;   // launched (0) or failed (< 0); 1: fall through
        }
        dim3 grid((unsigned)ncb, (unsigned)nchw);
        if (wide) {
            if (nj == 2) ec_xsum_kernel<CodeT, 2, 256><<<grid, 256, 0, stream>>>(X);
            else ec_xsum_kernel<CodeT, 1, 256><<<grid, 256, 0, stream>>>(X);
        } else {
            if (nj == 2) ec_xsum_kernel<CodeT, 2, 128><<<grid, 256, 0, stream>>>(X);
            else ec_xsum_kernel<CodeT, 1, 128><<<grid, 256, 0, stream>>>(X);
        }
        S3R_CHECK_LAUNCH();
    } else {
        for (int j = 0; j < nj; ++j) {
            dim3 grid((unsigned)s3r_cdiv(K, 128), (unsigned)nch);
            ec_xsum_partial_generic_kernel<<<grid, 128, 0, stream>>>(static_cast<const CodeT*>(X8), T, K,
                                                                    jobs[j].eps, xs, ps);
            S3R_CHECK_LAUNCH();
            ec_xsum_reduce_generic_kernel<<<(unsigned)s3r_cdiv(K, 256), 256, 0, stream>>>(
                xs, ps, nch, K, B, S / kXsumChunk, jobs[j].xsum, jobs[j].p);
            S3R_CHECK_LAUNCH();
        }
    }
    return S3R_OK;
}

// Checks and dispatch shared by the single-linear C entry point and the
// two-linear path of the FFN block.
static int ec_correct_jobs(const EcJob* jobs, int nj, int64_t T, int64_t N, int64_t S, int64_t K, const void* X8,
                           int code_format, int ec_mode, void* workspace, size_t workspace_bytes,
                           int* d_status, cudaStream_t stream) {
    if (T < 0 || N < 0 || K < 0 || S <= 0) return S3R_ERR_ARG;
    if (code_format != S3R_CODES_S8 && code_format != S3R_CODES_F16) return S3R_ERR_ARG;
    if (ec_mode != S3R_EC_NONE && ec_mode != S3R_EC_DX_ONLY && ec_mode != S3R_EC_TWO_WAY) return S3R_ERR_ARG;
    if (T == 0 || N == 0) return S3R_OK;
    if (T % S != 0) return S3R_ERR_SHAPE;
    if (S % kTile != 0 && S != T) return S3R_ERR_SHAPE;
    for (int j = 0; j < nj; ++j) {
        const EcJob& J = jobs[j];
        if (!J.tok || !J.col || !J.eps || !J.mu || !J.colmean) return S3R_ERR_ARG;
        if (ec_mode != S3R_EC_NONE && K > 0 && (!J.W8 || !J.rowsum || !J.v)) return S3R_ERR_ARG;
        if (ec_mode == S3R_EC_TWO_WAY && K > 0 && (!J.xsum || !J.p)) return S3R_ERR_ARG;
    }
    if (ec_mode == S3R_EC_TWO_WAY && K > 0 && !X8) return S3R_ERR_ARG;
    if (code_format == S3R_CODES_F16)
        return launch_factors<__half>(jobs, nj, T, N, S, K, X8, ec_mode, workspace, workspace_bytes, d_status,
                                      stream);
    return launch_factors<int8_t>(jobs, nj, T, N, S, K, X8, ec_mode, workspace, workspace_bytes, d_status, stream);
}

}  // namespace s3r

using namespace s3r;

extern "C" size_t s3r_ec_workspace_size(int64_t T, int64_t K) {
    if (T <= 0 || K <= 0) return 0;
    return xsum_workspace_bytes(T, K, 1);
}

extern "C" int s3r_ec_correct(const float* tok_err_part, const float* col_err_part, int64_t T, int64_t N, int64_t S,
                              const void* W8, int64_t K, const void* X8, int code_format, int ec_mode, float* eps,
                              float* mu, float* colmean, int32_t* rowsum, float* v, int32_t* xsum, float* p,
                              void* workspace, size_t workspace_bytes, int* d_status, cudaStream_t stream) {
    const EcJob job{tok_err_part, col_err_part, W8, eps, mu, colmean, rowsum, v, xsum, p};
    return ec_correct_jobs(&job, 1, T, N, S, K, X8, code_format, ec_mode, workspace, workspace_bytes, d_status,
                           stream);
}

// The two linears of the SwiGLU block that read the same input X (W1 and W3):
// the same factors as two s3r_ec_correct calls, bit for bit, in one pass.
size_t s3r_ec_pair_workspace_size(int64_t T, int64_t K) {
    if (T <= 0 || K <= 0) return 0;
    return xsum_workspace_bytes(T, K, 2);
}

int s3r_ec_correct_pair(const float* tok1, const float* col1, const void* W1_8, float* eps1, float* mu1,
                        float* colmean1, int32_t* rowsum1, float* v1, int32_t* xsum1, float* p1, const float* tok3,
                        const float* col3, const void* W3_8, float* eps3, float* mu3, float* colmean3,
                        int32_t* rowsum3, float* v3, int32_t* xsum3, float* p3, int64_t T, int64_t N, int64_t S,
                        int64_t K, const void* X8, int code_format, int ec_mode, void* workspace,
                        size_t workspace_bytes, int* d_status, cudaStream_t stream) {
    const EcJob jobs[2] = {{tok1, col1, W1_8, eps1, mu1, colmean1, rowsum1, v1, xsum1, p1},
                           {tok3, col3, W3_8, eps3, mu3, colmean3, rowsum3, v3, xsum3, p3}};
    return ec_correct_jobs(jobs, 2, T, N, S, K, X8, code_format, ec_mode, workspace, workspace_bytes, d_status,
                           stream);
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
// holds is written before it is read, and the column-block counters are
// zeroed by the first kernel of each call).  Calls that overlap on the GPU (two
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
