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
// (blockIdx.y selects the linear).  The first kMeansTokBlocks(T) blocks take
// eight tokens each, one warp per token: lane-strided sums over the token's
// tile partials (coalesced), then a butterfly; the rest take one (b, n) each,
// summing the example's tile rows in order.
constexpr int kMeansTokPerBlock = 8;
__host__ __device__ inline int64_t means_tok_blocks(int64_t T) { return (T + kMeansTokPerBlock - 1) / kMeansTokPerBlock; }
__global__ void __launch_bounds__(256) ec_means_kernel(EcMeansArgs A) {
    const int j = blockIdx.y;
    const float* tok = j ? A.tok[1] : A.tok[0];
    const float* col = j ? A.col[1] : A.col[0];
    float* eps = j ? A.eps[1] : A.eps[0];
    float* colmean = j ? A.colmean[1] : A.colmean[0];
    const int64_t T = A.T, N = A.N, S = A.S, B = T / S;
    if (A.counter && blockIdx.x == 0 && j == 0)
        for (int c = threadIdx.x; c < A.ncounter; c += blockDim.x) A.counter[c] = 0;
    const int64_t tb = means_tok_blocks(T);
    if ((int64_t)blockIdx.x < tb) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int64_t t = (int64_t)blockIdx.x * kMeansTokPerBlock + warp;
        if (t < T) {
            const float* row = tok + t * A.ntc;
            float s = 0.0f;
#pragma unroll 4
            for (int64_t c = lane; c < A.ntc; c += 32) s += row[c];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
            if (lane == 0) eps[t] = s / (float)N;
        }
    } else {
        const int64_t k = ((int64_t)blockIdx.x - tb) * blockDim.x + threadIdx.x;
        if (k < B * N) {
            const int64_t b = k / N, n = k % N;
            int64_t r_begin, r_end;
            if (B == 1) { r_begin = 0; r_end = A.ntr; }
            else { r_begin = b * (S / kTile); r_end = (b + 1) * (S / kTile); }
            float s = 0.0f;
#pragma unroll 8
            for (int64_t r = r_begin; r < r_end; ++r) s += col[r * N + n];
            colmean[b * N + n] = s / (float)S;
        }
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

// ---------------------------------------------------------------------------
// fp16 codes: the weight-side factors (rowsum, v) and the input-side factors
// (xsum, p) of up to two linears in one persistent launch that streams every
// code matrix through shared memory once.
//
// Work items, handed out in order by an atomic queue when the call has a
// workspace (gemv items first, the larger ones), else strided over the CTAs:
//   gemv (linear j, examples BCH g .. BCH g + BCH - 1, weight rows 32 rb ..
//     32 rb + 31): boxes of 32 rows x 256 channels of W8_j, each with the
//     matching BCH x 256 slab of colmean_j; consumer warp w keeps rows w and
//     w + 16, lane l channels 8 l .. 8 l + 7, and after the last box the
//     lanes meet in a reduce-scatter and the warp stores its two rows.  The
//     sums of codes are exact in fp32 (|sum| <= 127 N < 2^24).
//   xsum (256-column block cb, chunk c of XR rows of X8): XR / 64 boxes of
//     64 rows x 256 columns, each with the matching 64 entries of eps_j; warp
//     w takes rows w + 16 i, lane l columns 8 l .. 8 l + 7; after the last
//     box the 16 warps meet in shared memory (a written / read mbarrier pair)
//     and add their partials in warp order into the chunk's workspace row.
// Warp 16 is the producer.  One lane takes item ids from the queue one item
// ahead (the atomic's latency hides behind the copies), posts each id in a
// small ring before the item's first copy, and keeps kEsStages boxes in
// flight; a stage is refilled once all 16 consumer warps have released it.
// Consumer warps wait for every box on their own and never meet the producer
// in a CTA barrier.  Every wait is bounded and gives up early once another
// warp has raised the CTA's abort flag.  After a grid barrier (bounded) every
// thread of the grid takes a share of the fixed-order sums over the chunks.
// mu_b of every linear is computed by each CTA in the same fixed order (the
// same bits everywhere) while the first copies land.
// ---------------------------------------------------------------------------
constexpr int kEsConsumers = 16;                              // consumer warps
constexpr int kEsThreads = 32 * (kEsConsumers + 1);           // plus the producer warp
constexpr int kEsStages = 5;
constexpr int kEsXRowsBox = 64, kEsWRows = 32;
constexpr int kEsCmOff = kEsWRows * 256 * 2;             // colmean slab after the 16 KiB of weight codes
constexpr int kEsEpsOff = kEsXRowsBox * 256 * 2;         // eps slices after the 32 KiB of input codes
constexpr int kEsStageBytes = kEsEpsOff + kMaxJobs * kEsXRowsBox * 4;
constexpr int kEsQueue = 8;                              // item ids in flight per CTA
constexpr int kEsMaxB = 1024;                            // examples whose mu a CTA holds

// Dynamic shared memory: ring (128-byte aligned) | full and empty barriers of
// the stages, the exchange's two barriers | the exchange [16][(1 + nj) 256]
// floats | mu [nj][B].
static size_t es_smem_bytes(int nj, int64_t B) {
    return 128 + (size_t)kEsStages * kEsStageBytes + (2 * kEsStages + 2) * 8 +
           (size_t)kEsConsumers * 256 * (1 + nj) * 4 + (size_t)nj * (size_t)B * 4;
}

struct EcStreamArgs {
    int64_t T, K, N, S, B;
    const float* eps[kMaxJobs];
    float* mu[kMaxJobs];
    int32_t* rowsum[kMaxJobs];
    float* v[kMaxJobs];
    int32_t* xsum[kMaxJobs];
    float* p[kMaxJobs];
    int32_t* xs;       // [nch, K]
    float* ps;         // [NJ, nch, K]
    int* counter;      // the work queue (null: static assignment)
    int* done;         // grid barrier of the column-sum pass (null: no input-side items)
    int64_t ncb, nch;  // column blocks and chunks of the input-side pass
    int xr;            // rows per chunk (128, 256 or 512)
    int64_t ngr;       // weight row blocks per linear
    int ngroups;       // example groups of BCH
    int64_t nbn;       // channel boxes per weight row block
    int64_t n_gemv, n_items;
    int mu_v4;         // eps 16-byte aligned and S % 4 == 0: vector loads for mu
    int* d_status;
};

__device__ __forceinline__ void es_tma(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void es_tma1(uint32_t dst, const CUtensorMap* map, int32_t x, uint32_t bar) {
    es_tma(dst, map, x, 0, bar);
}
// A copy of streamed codes, read once: marked first to leave L2, so the chunk
// partials written meanwhile (and read back after the grid barrier) stay.
__device__ __forceinline__ void es_tma_stream(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, uint32_t bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3}], [%4], %5;" ::"r"(dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void es_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// the consumer warps' named barrier (the producer warp never takes part)
__device__ __forceinline__ void es_consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kEsConsumers) : "memory");
}
// Bounded wait (2 s of %globaltimer) that also gives up once the CTA's abort flag is up.
__device__ __forceinline__ bool es_wait(uint32_t bar, uint32_t parity, const volatile int* abort_flag,
                                        uint64_t limit_ns = 2000000000ull) {
    const uint64_t t0 = ec_gtime();
    while (true) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
        if (*abort_flag || ec_gtime() - t0 > limit_ns) return false;
    }
}

// Test hook: es_wait on a barrier that nothing arrives on, with a short limit;
// with raise_abort a second warp raises the CTA's abort flag after about a
// millisecond instead.  The waiter records how long it waited and sets
// S3R_ERR_TIMEOUT.
__global__ void __launch_bounds__(64) es_wait_probe_kernel(uint64_t limit_ns, int raise_abort, int* d_status,
                                                           unsigned long long* waited_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_s;
    const uint32_t b = (uint32_t)__cvta_generic_to_shared(&bar);
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b) : "memory");
        abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 32 && raise_abort) {
        const uint64_t t0 = ec_gtime();
        while (ec_gtime() - t0 < 1000000ull) {}
        *reinterpret_cast<volatile int*>(&abort_s) = 1;
    } else if (threadIdx.x == 0) {
        const uint64_t t0 = ec_gtime();
        const bool ok = es_wait(b, 0u, &abort_s, limit_ns);
        *waited_ns = ec_gtime() - t0;
        if (!ok) set_status(d_status, S3R_ERR_TIMEOUT);
    }
}


// mu[b] = (1/S) sum_{t < S} e[b S + t] for every b < B over the 512 consumer
// threads in a fixed order: per-thread strided sums (float4 loads when V4),
// a butterfly in each warp, then the 16 warps in order.  red holds 8 x 16 floats.
template <bool V4>
__device__ void es_mu(const float* e, int64_t S, int64_t B, float* red, float* out) {
    constexpr int NT = 32 * kEsConsumers;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int64_t b0 = 0; b0 < B; b0 += 8) {
        float s[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) s[q] = 0.0f;
        if (V4) {
#pragma unroll 2
            for (int64_t i = 4 * tid; i < S; i += 4 * NT) {
                float4 v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    v[q] = b0 + q < B ? __ldg(reinterpret_cast<const float4*>(e + (b0 + q) * S + i))
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int q = 0; q < 8; ++q) s[q] += (v[q].x + v[q].y) + (v[q].z + v[q].w);
            }
        } else {
#pragma unroll 4
            for (int64_t t = tid; t < S; t += NT) {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (b0 + q < B) s[q] += e[(b0 + q) * S + t];
            }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s[q] += __shfl_xor_sync(0xFFFFFFFFu, s[q], o);
            if (lane == 0) red[q * kEsConsumers + warp] = s[q];
        }
        es_consumers_sync();
        if (tid < 8 && b0 + tid < B) {
            float m = 0.0f;
#pragma unroll
            for (int w = 0; w < kEsConsumers; ++w) m += red[tid * kEsConsumers + w];
            out[b0 + tid] = m / (float)S;
        }
        es_consumers_sync();
    }
}

// V = 2^m values per lane (V <= 32) summed over the warp: a reduce-scatter
// (halving exchanges) then plain exchanges, in a fixed order.  Returns, in
// every lane, the full sum of value lane / (32 / V).
template <int V>
__device__ __forceinline__ float warp_scatter(const float (&v)[V]) {
    const int lane = threadIdx.x & 31;
    float a[V];
#pragma unroll
    for (int i = 0; i < V; ++i) a[i] = v[i];
    int n = V;
#pragma unroll
    for (int x = 16; x >= 1; x >>= 1) {
        if (n > 1) {
            const int h = n / 2;
            const bool hi = lane & x;
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
                if (i < h) {
                    const float send = hi ? a[i] : a[i + h], keep = hi ? a[i + h] : a[i];
                    a[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, x);
                }
            }
            n = h;
        } else {
            a[0] += __shfl_xor_sync(0xFFFFFFFFu, a[0], x);
        }
    }
    return a[0];
}

template <int NJ, int BCH>
__global__ void __launch_bounds__(kEsThreads, 1)
    ec_stream_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW0,
                     const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmC0,
                     const __grid_constant__ CUtensorMap tmC1, const __grid_constant__ CUtensorMap tmE0,
                     const __grid_constant__ CUtensorMap tmE1, EcStreamArgs A) {
    constexpr int NA = 1 + NJ;   // column-sum arrays: xs, then ps of each linear
    extern __shared__ uint8_t es_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(es_raw) + 127) & ~(uintptr_t)127);
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + kEsStages * kEsStageBytes);   // copies landed
    uint64_t* empty = full + kEsStages;                                                // consumers done
    uint64_t* xbar = empty + kEsStages;   // exchange: [0] partials written, [1] partials read
    float* red = reinterpret_cast<float*>(xbar + 2);              // [16][NA][256]
    float* mu_s = red + kEsConsumers * NA * 256;                  // [NJ][B]
    __shared__ float mred[8 * kEsConsumers];
    __shared__ int q_item[kEsQueue];
    __shared__ int last;
    __shared__ int abort_s;
    volatile int* abort_flag = &abort_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t K = A.K, B = A.B;
    const uint32_t bar0 = (uint32_t)__cvta_generic_to_shared(full);
    const uint32_t ebar0 = (uint32_t)__cvta_generic_to_shared(empty);
    const uint32_t xbar0 = (uint32_t)__cvta_generic_to_shared(xbar);
    const int n_items = (int)A.n_items, n_gemv = (int)A.n_gemv, ngr = (int)A.ngr, ncb = (int)A.ncb;
    const int per_j = ngr * A.ngroups;
    if (tid == 0) {
        for (int i = 0; i < kEsStages; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar0 + 8 * i) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(ebar0 + 8 * i), "n"(kEsConsumers) : "memory");
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(xbar0), "n"(kEsConsumers) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(xbar0 + 8), "n"(kEsConsumers) : "memory");
        abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    bool failed = false;
    int issued = 0;   // boxes (and the end mark) issued: the producer lane's count
    if (warp == kEsConsumers) {
        // ---- producer (one lane) ----
        if (lane == 0) {
            const CUtensorMap* maps[7] = {&tmX, &tmW0, &tmW1, &tmC0, &tmC1, &tmE0, &tmE1};
            for (int i = 0; i < 7; ++i) asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)maps[i]) : "memory");
            int p_fetched = 0;
            auto fetch = [&]() -> int {
                const int it = A.counter ? atomicAdd(A.counter, 1) : (int)blockIdx.x + p_fetched * (int)gridDim.x;
                ++p_fetched;
                return it < n_items ? it : -1;
            };
            uint64_t evict_first;
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(evict_first));
            int p_next = fetch(), p_box = 0, p_nbox = 0, p_ord = 0;
            bool p_gemv = false;
            const CUtensorMap *p_m0 = nullptr, *p_m1 = nullptr;
            int32_t p_x = 0, p_y = 0, p_y1 = 0;
            while (true) {
                const int s = issued % kEsStages;
                if (issued >= kEsStages) {
                    if (!es_wait(ebar0 + 8 * s, (uint32_t)(((issued / kEsStages) - 1) & 1), abort_flag)) {
                        failed = true;
                        break;
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                const uint32_t bar = bar0 + 8 * s;
                uint8_t* dst = ring + s * kEsStageBytes;
                if (p_box == p_nbox) {   // the next item, or the end mark
                    const int item = p_next;
                    q_item[p_ord % kEsQueue] = item;
                    ++p_ord;
                    p_box = 0;
                    if (item < 0) {
                        es_arrive(bar);
                        ++issued;
                        break;
                    }
                    p_next = fetch();
                    p_gemv = item < n_gemv;
                    if (p_gemv) {
                        const int j = item / per_j, rem = item - j * per_j;
                        const int g = rem / ngr, rb = rem - g * ngr;
                        p_m0 = j ? &tmW1 : &tmW0;
                        p_m1 = j ? &tmC1 : &tmC0;
                        p_y = rb * kEsWRows;
                        p_y1 = g * BCH;
                        p_nbox = (int)A.nbn;
                    } else {
                        const int xi = item - n_gemv, c = xi / ncb, cb = xi - c * ncb;
                        p_x = cb * 256;
                        p_y = c * A.xr;
                        p_nbox = A.xr / kEsXRowsBox;
                    }
                }
                if (p_gemv) {
                    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                                 "r"(kEsCmOff + BCH * 256 * 4)
                                 : "memory");
                    es_tma_stream((uint32_t)__cvta_generic_to_shared(dst), p_m0, p_box * 256, p_y, bar, evict_first);
                    es_tma((uint32_t)__cvta_generic_to_shared(dst + kEsCmOff), p_m1, p_box * 256, p_y1, bar);
                } else {
                    const int32_t y = p_y + p_box * kEsXRowsBox;
                    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                                 "r"(kEsEpsOff + NJ * kEsXRowsBox * 4)
                                 : "memory");
                    es_tma_stream((uint32_t)__cvta_generic_to_shared(dst), &tmX, p_x, y, bar, evict_first);
                    es_tma1((uint32_t)__cvta_generic_to_shared(dst + kEsEpsOff), &tmE0, y, bar);
                    if (NJ > 1)
                        es_tma1((uint32_t)__cvta_generic_to_shared(dst + kEsEpsOff + kEsXRowsBox * 4), &tmE1, y, bar);
                }
                ++p_box;
                ++issued;
            }
        }
    } else {
        // ---- consumers ----
        for (int j = 0; j < NJ; ++j) {
            if (A.mu_v4) es_mu<true>(A.eps[j], A.S, B, mred, mu_s + j * B);
            else es_mu<false>(A.eps[j], A.S, B, mred, mu_s + j * B);
        }
        if (blockIdx.x == 0)
            for (int j = 0; j < NJ; ++j)
                for (int64_t b = tid; b < B; b += 32 * kEsConsumers) A.mu[j][b] = mu_s[j * B + b];
        int k = 0;    // boxes consumed
        int ord = 0;  // items consumed
        int nx = 0;   // input-side items consumed (phases of the exchange)
        auto release = [&]() {
            __syncwarp();
            if (lane == 0) es_arrive(ebar0 + 8 * (k % kEsStages));
            ++k;
        };
        while (!failed) {
            if (!es_wait(bar0 + 8 * (k % kEsStages), (uint32_t)((k / kEsStages) & 1), abort_flag)) {
                failed = true;
                break;
            }
            const int item = q_item[ord % kEsQueue];
            if (item < 0) break;   // the end mark (no copy behind it, no refill after it)
            ++ord;
            if (item < n_gemv) {
                const int j = item / per_j, rem = item - j * per_j;
                const int g = rem / ngr;
                const int64_t rb = rem - g * ngr;
                const float* mu_j = mu_s + j * B;
                // accumulators over channel pairs (2e, 2e + 1), one per row and example
                float2 acc[2][BCH], rs[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    rs[i] = make_float2(0.0f, 0.0f);
#pragma unroll
                    for (int q = 0; q < BCH; ++q) acc[i][q] = make_float2(0.0f, 0.0f);
                }
                for (int bx = 0; bx < (int)A.nbn; ++bx) {
                    if (bx > 0 && !es_wait(bar0 + 8 * (k % kEsStages), (uint32_t)((k / kEsStages) & 1), abort_flag)) {
                        failed = true;
                        break;
                    }
                    const uint8_t* st = ring + (k % kEsStages) * kEsStageBytes;
                    float2 x2[2][4];
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const uint4 w = *reinterpret_cast<const uint4*>(st + ((warp + 16 * i) * 256 + 8 * lane) * 2);
                        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            x2[i][e] = __half22float2(*reinterpret_cast<const __half2*>(&u[e]));
                            rs[i] = f2_add(rs[i], x2[i][e]);
                        }
                    }
                    // centered channel means of my 8 channels, one example at a time (past N and
                    // past B the copies read zero)
#pragma unroll
                    for (int q = 0; q < BCH; ++q) {
                        const int64_t b = (int64_t)g * BCH + q;
                        const float m = b < B ? mu_j[b] : 0.0f;
                        const float2 m2 = make_float2(m, m);
                        const float4 c0 = *reinterpret_cast<const float4*>(st + kEsCmOff + (q * 256 + 8 * lane) * 4);
                        const float4 c1 =
                            *reinterpret_cast<const float4*>(st + kEsCmOff + (q * 256 + 8 * lane + 4) * 4);
                        const float2 cm2[4] = {f2_sub(make_float2(c0.x, c0.y), m2), f2_sub(make_float2(c0.z, c0.w), m2),
                                               f2_sub(make_float2(c1.x, c1.y), m2), f2_sub(make_float2(c1.z, c1.w), m2)};
#pragma unroll
                        for (int i = 0; i < 2; ++i)
#pragma unroll
                            for (int e = 0; e < 4; ++e) acc[i][q] = f2_fma(cm2[e], x2[i][e], acc[i][q]);
                    }
                    release();
                }
                if (failed) break;
                // row sums: integers, one reduction each; v: a reduce-scatter of the 2 x BCH values,
                // after which lane l holds value l / (32 / (2 BCH)) = (row, example) in row-major order
                int ri[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) ri[i] = __reduce_add_sync(0xFFFFFFFFu, (int)(rs[i].x + rs[i].y));
                float vv[2 * BCH];
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int q = 0; q < BCH; ++q) vv[i * BCH + q] = acc[i][q].x + acc[i][q].y;
                const float vsum = warp_scatter<2 * BCH>(vv);
                constexpr int G = 32 / (2 * BCH);   // lanes per value
                const int vi = lane / G, i = vi / BCH, q = vi - i * BCH;
                const int64_t kr = rb * kEsWRows + warp + 16 * i;
                const int64_t b = (int64_t)g * BCH + q;
                if (lane % G == 0 && kr < K && b < B) A.v[j][b * K + kr] = vsum;
                if (lane < 2 && g == 0) {
                    const int64_t kr2 = rb * kEsWRows + warp + 16 * lane;
                    if (kr2 < K) A.rowsum[j][kr2] = lane ? ri[1] : ri[0];
                }
            } else {
                const int xi = item - n_gemv;
                const int64_t c = xi / ncb, cb = xi - c * ncb;
                float2 sx[4], sp[NJ][4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    sx[q] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int jj = 0; jj < NJ; ++jj) sp[jj][q] = make_float2(0.f, 0.f);
                }
                const int nb = A.xr / kEsXRowsBox;
                for (int bx = 0; bx < nb; ++bx) {
                    if (bx > 0 && !es_wait(bar0 + 8 * (k % kEsStages), (uint32_t)((k / kEsStages) & 1), abort_flag)) {
                        failed = true;
                        break;
                    }
                    const uint8_t* st = ring + (k % kEsStages) * kEsStageBytes;
                    const float* es = reinterpret_cast<const float*>(st + kEsEpsOff);   // zero past T
#pragma unroll
                    for (int i = 0; i < kEsXRowsBox / kEsConsumers; ++i) {
                        const int r = warp + kEsConsumers * i;
                        const uint4 w = *reinterpret_cast<const uint4*>(st + (r * 256 + 8 * lane) * 2);
                        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
                        float e[NJ];
#pragma unroll
                        for (int jj = 0; jj < NJ; ++jj) e[jj] = es[jj * kEsXRowsBox + r];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&u[q]));
                            sx[q] = f2_add(sx[q], x);
#pragma unroll
                            for (int jj = 0; jj < NJ; ++jj)
                                sp[jj][q] = f2_fma(x, make_float2(e[jj], e[jj]), sp[jj][q]);
                        }
                    }
                    release();
                }
                if (failed) break;
                // the chunk's column sums: the 16 warps meet in shared memory and add up in warp order
                if (nx > 0 && !es_wait(xbar0 + 8, (uint32_t)((nx - 1) & 1), abort_flag)) {   // last item's sums read
                    failed = true;
                    break;
                }
                {
                    float* mine = red + warp * NA * 256 + 8 * lane;
                    *reinterpret_cast<float4*>(mine) = make_float4(sx[0].x, sx[0].y, sx[1].x, sx[1].y);
                    *reinterpret_cast<float4*>(mine + 4) = make_float4(sx[2].x, sx[2].y, sx[3].x, sx[3].y);
#pragma unroll
                    for (int jj = 0; jj < NJ; ++jj) {
                        float* pj = mine + (1 + jj) * 256;
                        *reinterpret_cast<float4*>(pj) = make_float4(sp[jj][0].x, sp[jj][0].y, sp[jj][1].x, sp[jj][1].y);
                        *reinterpret_cast<float4*>(pj + 4) =
                            make_float4(sp[jj][2].x, sp[jj][2].y, sp[jj][3].x, sp[jj][3].y);
                    }
                }
                __syncwarp();
                if (lane == 0) es_arrive(xbar0);
                if (!es_wait(xbar0, (uint32_t)(nx & 1), abort_flag)) {   // every warp's partials written
                    failed = true;
                    break;
                }
                for (int vi = tid; vi < NA * 256; vi += 32 * kEsConsumers) {
                    const int a = vi >> 8, col = vi & 255;
                    float sum = 0.0f;
#pragma unroll
                    for (int w = 0; w < kEsConsumers; ++w) sum += red[(w * NA + a) * 256 + col];
                    const int64_t kcol = cb * 256 + col;
                    if (kcol < K) {
                        if (a == 0) A.xs[c * K + kcol] = (int32_t)sum;
                        else A.ps[((int64_t)(a - 1) * A.nch + c) * K + kcol] = sum;
                    }
                }
                __syncwarp();
                if (lane == 0) es_arrive(xbar0 + 8);
                ++nx;
            }
        }
    }
    if (failed) {
        *abort_flag = 1;
        if (A.d_status) *(volatile int*)A.d_status = S3R_ERR_TIMEOUT;
    }
    __syncthreads();
    if (A.done) {
        // Every CTA of the (cooperative, co-resident) grid has written its chunk
        // partials: meet at a grid barrier (one counter, bounded wait), then
        // every thread of the grid adds up its share of the chunks in a fixed order.
        if (tid == 0) {
            __threadfence();
            atomicAdd(A.done, 1);
            const uint64_t t0 = ec_gtime();
            bool met = false;
            while (!met) {
                int v;
                asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(A.done) : "memory");
                met = v >= (int)gridDim.x;
                if (!met && ec_gtime() - t0 > 2000000000ull) break;
            }
            last = met && !*abort_flag;
            if (!met && A.d_status) *(volatile int*)A.d_status = S3R_ERR_TIMEOUT;
        }
        __syncthreads();
        if (last) {
            __threadfence();
            const int64_t cpe = B == 1 ? A.nch : A.S / A.xr;   // chunks per example
            const int64_t gthreads = (int64_t)gridDim.x * kEsThreads;
            const int64_t gtid = (int64_t)blockIdx.x * kEsThreads + tid;
            if (B <= 32 && (B & (B - 1)) == 0) {
                // a warp takes 32 / B columns, one lane per (column, example): the example's
                // chunks in order, then p over the B lanes of the column in a butterfly
                const int cpw = 32 / (int)B;
                const int64_t nwarps = gthreads >> 5;
                const int b = lane % (int)B;
                for (int64_t base = (gtid >> 5) * cpw; base < K; base += nwarps * cpw) {
                    const int64_t kcol = base + lane / (int)B;
                    const bool on = kcol < K;
                    int xb = 0;
                    float pb[NJ];
#pragma unroll
                    for (int jj = 0; jj < NJ; ++jj) pb[jj] = 0.0f;
                    if (on) {
#pragma unroll 8
                        for (int64_t cc = b * cpe; cc < (b + 1) * cpe; ++cc) {
                            xb += __ldcg(A.xs + cc * K + kcol);
#pragma unroll
                            for (int jj = 0; jj < NJ; ++jj) pb[jj] += __ldcg(A.ps + (jj * A.nch + cc) * K + kcol);
                        }
#pragma unroll
                        for (int jj = 0; jj < NJ; ++jj) A.xsum[jj][b * K + kcol] = xb;
                    }
                    for (int o = (int)B / 2; o >= 1; o >>= 1)
#pragma unroll
                        for (int jj = 0; jj < NJ; ++jj) pb[jj] += __shfl_xor_sync(0xFFFFFFFFu, pb[jj], o);
                    if (on && b == 0)
#pragma unroll
                        for (int jj = 0; jj < NJ; ++jj) A.p[jj][kcol] = pb[jj];
                }
            } else {
                for (int64_t kcol = gtid; kcol < K; kcol += gthreads) {
                    float pk[NJ];
#pragma unroll
                    for (int jj = 0; jj < NJ; ++jj) pk[jj] = 0.0f;
                    for (int64_t b2 = 0; b2 < B; ++b2) {
                        int xbi = 0;
                        float pb[NJ];
#pragma unroll
                        for (int jj = 0; jj < NJ; ++jj) pb[jj] = 0.0f;
#pragma unroll 8
                        for (int64_t cc = b2 * cpe; cc < (b2 + 1) * cpe; ++cc) {
                            xbi += __ldcg(A.xs + cc * K + kcol);
#pragma unroll
                            for (int jj = 0; jj < NJ; ++jj) pb[jj] += __ldcg(A.ps + (jj * A.nch + cc) * K + kcol);
                        }
#pragma unroll
                        for (int jj = 0; jj < NJ; ++jj) {
                            A.xsum[jj][b2 * K + kcol] = xbi;
                            pk[jj] += pb[jj];
                        }
                    }
#pragma unroll
                    for (int jj = 0; jj < NJ; ++jj) A.p[jj][kcol] = pk[jj];
                }
            }
        }
    }
    // an early exit may leave copies in flight: the producer waits for them before leaving
    if (*abort_flag && warp == kEsConsumers && lane == 0)
        for (int q = issued > kEsStages ? issued - kEsStages : 0; q < issued; ++q)
            xs_wait(bar0 + 8 * (q % kEsStages), (uint32_t)((q / kEsStages) & 1));
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

static int ec_sm_count() { return s3r_sm_count(); }

// max_ctas > 0 caps the grid (a call that shares the GPU with other such calls
// on other streams takes its share of the SMs instead of all of them).
template <int NJ, int BCH>
static int launch_ec_stream_t(const CUtensorMap* maps, const EcStreamArgs& S, size_t smem, int max_ctas,
                              cudaStream_t stream) {
    const int st = s3r_kernel_smem((const void*)ec_stream_kernel<NJ, BCH>, (int)es_smem_bytes(NJ, kEsMaxB),
                                   "ec stream: cudaFuncSetAttribute");
    if (st) return st;
    int64_t grid = std::min<int64_t>(S.n_items, ec_sm_count());
    if (max_ctas > 0) grid = std::min<int64_t>(grid, max_ctas);
    if (!S.done) {
        ec_stream_kernel<NJ, BCH><<<(unsigned)grid, kEsThreads, smem, stream>>>(maps[0], maps[1], maps[2], maps[3],
                                                                                 maps[4], maps[5], maps[6], S);
        S3R_CHECK_LAUNCH();
        return S3R_OK;
    }
    // the column-sum pass ends with a grid barrier: a cooperative launch keeps every CTA resident
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ec_stream_kernel<NJ, BCH>, kEsThreads, smem) !=
            cudaSuccess ||
        per_sm < 1) {
        (void)cudaGetLastError();
        return 1;
    }
    grid = std::min<int64_t>(grid, (int64_t)per_sm * ec_sm_count());
    EcStreamArgs a = S;
    CUtensorMap m[7];
    for (int i = 0; i < 7; ++i) m[i] = maps[i];
    void* args[8] = {&m[0], &m[1], &m[2], &m[3], &m[4], &m[5], &m[6], &a};
    const cudaError_t e = cudaLaunchCooperativeKernel((const void*)ec_stream_kernel<NJ, BCH>, dim3((unsigned)grid),
                                                      dim3(kEsThreads), args, smem, stream);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return s3r_cuda_fail("ec stream: cudaLaunchCooperativeKernel", e);
    }
    s3r_count_launch();
    return S3R_OK;
}

static int launch_ec_stream(const EcJob* jobs, int nj, int64_t T, int64_t N, int64_t S, int64_t K, const void* X8,
                            bool weight, bool two, int32_t* xs, float* ps, int* counter, int max_ctas,
                            int* d_status, cudaStream_t stream) {
    const int64_t B = T / S;
    if (B > kEsMaxB || T >= (int64_t(1) << 31) || K >= (int64_t(1) << 31) || N >= (int64_t(1) << 31)) return 1;
    if (N % 8 != 0 || (two && K % 8 != 0)) return 1;
    for (int j = 0; j < nj; ++j)
        if ((weight && (!s3r_aligned16(jobs[j].W8) || !s3r_aligned16(jobs[j].colmean))) ||
            (two && !s3r_aligned16(jobs[j].eps)))
            return 1;
    if (two && !s3r_aligned16(X8)) return 1;
    auto fn = ec_encode_fn();
    if (!fn) return 1;
    const int bch = B == 1 ? 1 : (B <= 4 ? 4 : 8);
    CUtensorMap maps[7];
    const cuuint32_t estr[2] = {1, 1};
    auto enc2 = [&](CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows,
                    uint64_t pitch_bytes, uint32_t bc, uint32_t br) {
        const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
        const cuuint64_t strides[1] = {(cuuint64_t)pitch_bytes};
        const cuuint32_t box[2] = {bc, br};
        return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    // a vector as one row of a 2-D map (entries past n read as zero)
    auto enc1 = [&](CUtensorMap* m, const float* base, uint64_t n) {
        return enc2(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, n, 1, (n * 4 + 15) / 16 * 16, kEsXRowsBox, 1);
    };
    for (int j = 0; j < nj; ++j) {
        if (weight &&
            (!enc2(&maps[1 + j], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, jobs[j].W8, N, K, N * 2, 256, kEsWRows) ||
             !enc2(&maps[3 + j], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, jobs[j].colmean, N, B, N * 4, 256, bch)))
            return 1;
        if (two && !enc1(&maps[5 + j], jobs[j].eps, T)) return 1;
    }
    if (two) {
        if (!enc2(&maps[0], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, X8, K, T, K * 2, 256, kEsXRowsBox)) return 1;
    } else {
        maps[0] = maps[1];   // not read without input-side items
        maps[5] = maps[1];
    }
    if (!weight)
        for (int j = 0; j < 2; ++j) {   // not read without weight-side items
            maps[1 + j] = maps[0];
            maps[3 + j] = maps[0];
        }
    if (nj == 1) {
        maps[2] = maps[1];
        maps[4] = maps[3];
        maps[6] = maps[5];
    }
    if (!two) maps[6] = maps[5];
    EcStreamArgs A{};
    A.T = T; A.K = K; A.N = N; A.S = S; A.B = B;
    for (int j = 0; j < nj; ++j) {
        A.eps[j] = jobs[j].eps;
        A.mu[j] = jobs[j].mu;
        A.rowsum[j] = jobs[j].rowsum;
        A.v[j] = jobs[j].v;
        A.xsum[j] = jobs[j].xsum;
        A.p[j] = jobs[j].p;
    }
    A.xs = xs; A.ps = ps;
    A.counter = two ? counter + s3r_cdiv(K, 256) : nullptr;   // after the column-block counters of the other path
    A.done = two ? A.counter + 1 : nullptr;
    A.xr = (B == 1 || S % 512 == 0) ? 512 : (S % 256 == 0 ? 256 : 128);
    A.ncb = s3r_cdiv(K, 256);
    A.nch = s3r_cdiv(T, A.xr);
    A.ngr = s3r_cdiv(K, kEsWRows);
    A.ngroups = (int)s3r_cdiv(B, bch);
    A.nbn = s3r_cdiv(N, 256);
    A.n_gemv = weight ? nj * A.ngr * A.ngroups : 0;
    A.n_items = A.n_gemv + (two ? A.ncb * A.nch : 0);
    A.d_status = d_status;
    A.mu_v4 = S % 4 == 0;
    for (int j = 0; j < nj; ++j) A.mu_v4 = A.mu_v4 && s3r_aligned16(jobs[j].eps);
    if (A.n_items >= (int64_t(1) << 30)) return 1;
    const size_t smem = es_smem_bytes(nj, B);
    if (nj == 2) {
        if (bch == 1) return launch_ec_stream_t<2, 1>(maps, A, smem, max_ctas, stream);
        if (bch == 4) return launch_ec_stream_t<2, 4>(maps, A, smem, max_ctas, stream);
        return launch_ec_stream_t<2, 8>(maps, A, smem, max_ctas, stream);
    }
    if (bch == 1) return launch_ec_stream_t<1, 1>(maps, A, smem, max_ctas, stream);
    if (bch == 4) return launch_ec_stream_t<1, 4>(maps, A, smem, max_ctas, stream);
    return launch_ec_stream_t<1, 8>(maps, A, smem, max_ctas, stream);
}

// Workspace of the column-sum pass for `njobs` linears sharing X8 [T, K].
static size_t xsum_workspace_bytes(int64_t T, int64_t K, int njobs) {
    const size_t nch = (size_t)s3r_cdiv(T, kXsumChunk);   // the generic path's chunks, the finer of the two
    return nch * (size_t)K * (sizeof(int32_t) + njobs * sizeof(float)) + (size_t)s3r_cdiv(K, 256) * sizeof(int) +
           512;
}

template <typename CodeT>
static int launch_factors(const EcJob* jobs, int nj, int64_t T, int64_t N, int64_t S, int64_t K, const void* X8,
                          int ec_mode, void* workspace, size_t workspace_bytes, int max_ctas, int* d_status,
                          cudaStream_t stream) {
    const int64_t B = T / S, ntc = s3r_cdiv(N, kTile), ntr = s3r_cdiv(T, kTile);
    const bool two = ec_mode == S3R_EC_TWO_WAY || ec_mode == S3R_EC_DW_ONLY;     // input side: xsum, p
    const bool weight = ec_mode == S3R_EC_DX_ONLY || ec_mode == S3R_EC_TWO_WAY;  // weight side: rowsum, v
    bool vec_w = N % 8 == 0;
    for (int j = 0; j < nj; ++j) vec_w = vec_w && s3r_aligned16(jobs[j].W8) && s3r_aligned16(jobs[j].colmean);
    const int64_t slab = std::min<int64_t>(N, kGemvSlabFloats / kGemvBch);   // multiple of 8 when N is
    const size_t gsm = gemv_smem_bytes(slab, B);
    vec_w = vec_w && gsm <= 200 * 1024;
    // every warp holds at most kGemvPairs row pairs: one CTA per SM gives sms * kGemvWarps warps per launch
    const int gsms = s3r_sm_count();
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
        M.counter = two ? counter : nullptr;
        M.ncounter = (int)ncb + 2;   // the column blocks, then the streaming kernel's work queue and grid barrier
        dim3 grid((unsigned)(means_tok_blocks(T) + s3r_cdiv(B * N, 256)), (unsigned)nj);
        ec_means_kernel<<<grid, 256, 0, stream>>>(M);
        S3R_CHECK_LAUNCH();
    }
    if (ec_mode != S3R_EC_NONE && K > 0 && sizeof(CodeT) == 2) {
        const int st =
            launch_ec_stream(jobs, nj, T, N, S, K, X8, weight, two, xs, ps, counter, max_ctas, d_status, stream);
        if (st <= 0) return st;   // launched (0) or failed (< 0); 1: the kernels below
    }
    if (ec_mode == S3R_EC_NONE || K == 0 || !vec_w || !weight) {
        for (int j = 0; j < nj; ++j) {
            ec_mu_kernel<<<(unsigned)s3r_cdiv(B, 8), kGemvThreads, 0, stream>>>(jobs[j].eps, S, B, jobs[j].mu);
            S3R_CHECK_LAUNCH();
        }
    }
    if (ec_mode == S3R_EC_NONE || K == 0) return S3R_OK;
    if (!weight) {
    } else if (vec_w) {
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
        const int st = s3r_kernel_smem((const void*)ec_gemv_kernel<CodeT>, 200 * 1024, "ec gemv: cudaFuncSetAttribute");
        if (st) return st;
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
                           int* d_status, cudaStream_t stream, int max_ctas = 0) {
    if (T < 0 || N < 0 || K < 0 || S <= 0) return S3R_ERR_ARG;
    if (code_format != S3R_CODES_S8 && code_format != S3R_CODES_F16) return S3R_ERR_ARG;
    if (ec_mode < S3R_EC_NONE || ec_mode > S3R_EC_DW_ONLY) return S3R_ERR_ARG;
    const bool weight = ec_mode == S3R_EC_DX_ONLY || ec_mode == S3R_EC_TWO_WAY;   // rowsum and v
    const bool input = ec_mode == S3R_EC_TWO_WAY || ec_mode == S3R_EC_DW_ONLY;    // xsum and p
    if (T == 0 || N == 0) return S3R_OK;
    if (T % S != 0) return S3R_ERR_SHAPE;
    if (S % kTile != 0 && S != T) return S3R_ERR_SHAPE;
    for (int j = 0; j < nj; ++j) {
        const EcJob& J = jobs[j];
        if (!J.tok || !J.col || !J.eps || !J.mu || !J.colmean) return S3R_ERR_ARG;
        if (weight && K > 0 && (!J.W8 || !J.rowsum || !J.v)) return S3R_ERR_ARG;
        if (input && K > 0 && (!J.xsum || !J.p)) return S3R_ERR_ARG;
    }
    if (input && K > 0 && !X8) return S3R_ERR_ARG;
    if (code_format == S3R_CODES_F16)
        return launch_factors<__half>(jobs, nj, T, N, S, K, X8, ec_mode, workspace, workspace_bytes, max_ctas,
                                      d_status, stream);
    return launch_factors<int8_t>(jobs, nj, T, N, S, K, X8, ec_mode, workspace, workspace_bytes, max_ctas, d_status,
                                  stream);
}

}  // namespace s3r

using namespace s3r;

int ec_wait_probe(uint64_t limit_ns, int raise_abort, int* d_status, unsigned long long* waited_ns,
                  cudaStream_t stream) {
    es_wait_probe_kernel<<<1, 64, 0, stream>>>(limit_ns, raise_abort, d_status, waited_ns);
    S3R_CHECK_LAUNCH();
    return S3R_OK;
}

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

int s3r_ec_correct_capped(const float* tok_err_part, const float* col_err_part, int64_t T, int64_t N, int64_t S,
                          const void* W8, int64_t K, const void* X8, int code_format, int ec_mode, float* eps,
                          float* mu, float* colmean, int32_t* rowsum, float* v, int32_t* xsum, float* p,
                          void* workspace, size_t workspace_bytes, int max_ctas, int* d_status,
                          cudaStream_t stream) {
    const EcJob job{tok_err_part, col_err_part, W8, eps, mu, colmean, rowsum, v, xsum, p};
    return ec_correct_jobs(&job, 1, T, N, S, K, X8, code_format, ec_mode, workspace, workspace_bytes, d_status,
                           stream, max_ctas);
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
                        size_t workspace_bytes, int max_ctas, int* d_status, cudaStream_t stream) {
    const EcJob jobs[2] = {{tok1, col1, W1_8, eps1, mu1, colmean1, rowsum1, v1, xsum1, p1},
                           {tok3, col3, W3_8, eps3, mu3, colmean3, rowsum3, v3, xsum3, p3}};
    return ec_correct_jobs(jobs, 2, T, N, S, K, X8, code_format, ec_mode, workspace, workspace_bytes, d_status,
                           stream, max_ctas);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of s3r_ec_correct.
//
// Some callers cannot allocate device memory at the moment they run the
// backward: code running from a host callback or a real-time loop, where an
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
    if (ec_mode != S3R_EC_TWO_WAY && ec_mode != S3R_EC_DW_ONLY)   // only the column sums need scratch
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
