// gemm_mma.cu -- INT8 backward GEMMs on the warp-level s8 tensor-core path
// (mma.sync m16n8k32 s8 x s8 -> s32), with the per-128-K-block rescale and the
// S3R-EC epilogues.
//
// Paper: "Efficient Quantization Training with Stochastic Rounding via
// Structured Subspace Randomness" §III-A: S8 GEMM with S32 accumulation, then
// rescale; §III-D: subtract the image of P(E) through each product.
//
// Both products are run as C[m, n] = sum_kb scale(kb) * sum_{k in kb} A[m,k] B[n,k]
// with A and B row-major over the contraction index ("TN").  dX uses Q and W8
// directly; dW first transposes X8 and Q into the caller's workspace so that
// the token index is contiguous.  The int32 partial of every 128-wide block is
// exact and is promoted to fp32 with one fma per block, in ascending order.
#include "common.cuh"

namespace s3r {

constexpr int kBM = 128, kBN = 128, kBK = 128;
constexpr int kPitch = kBK + 16;  // bytes per smem row: 144 keeps fragment loads conflict-free
constexpr int kStageBytes = (kBM + kBN) * kPitch;
constexpr int kGemmSmem = 2 * kStageBytes;

enum Epi { kEpiDX = 0, kEpiDW = 1, kEpiDump = 2 };

struct GemmOperands {
    const int8_t* A;
    int64_t lda;
    const int8_t* B;
    int64_t ldb;
    int64_t M, N, K;
    const float* scale;  // scale(mt, nt, kb) = scale[mt*sm + nt*sn + kb*sk]
    int64_t sm, sn, sk;
    bool aligned;        // base pointers and row strides 16-byte aligned: cp.async path
};

struct GemmEpilogue {
    float* C;
    int64_t ldc;
    int32_t* dump;
    // dX
    const float* s_x;
    const float* eps;
    const int32_t* rowsum;
    const float* v;
    int accumulate;
    // dW
    const float* s_w;
    const float* colmean;
    const float* mu;
    const int32_t* xsum;
    const float* p;
    int ec_mode;
    int64_t S;
    int64_t B;
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void mma_s8(int32_t (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Stage one 128x128-byte block of A and of B into shared memory (zero-filled
// outside the matrices).
__device__ __forceinline__ void load_stage(const GemmOperands& P, int8_t* sA, int8_t* sB, int64_t m0, int64_t n0,
                                           int64_t k0) {
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int id = threadIdx.x + 256 * it;
        const int row = id >> 3, chunk = id & 7;
        const int64_t k = k0 + 16 * chunk;
        const int64_t rem = P.K - k;
        const int bytes_k = rem >= 16 ? 16 : (rem > 0 ? (int)rem : 0);
        const int64_t m = m0 + row, n = n0 + row;
        const bool okA = m < P.M && bytes_k > 0, okB = n < P.N && bytes_k > 0;
        if (P.aligned) {
            cp_async16(sA + row * kPitch + 16 * chunk, okA ? P.A + m * P.lda + k : P.A, okA ? bytes_k : 0);
            cp_async16(sB + row * kPitch + 16 * chunk, okB ? P.B + n * P.ldb + k : P.B, okB ? bytes_k : 0);
        } else {
            // unaligned rows: plain byte loads (correct for any stride, slower)
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                sA[row * kPitch + 16 * chunk + i] = (okA && i < bytes_k) ? P.A[m * P.lda + k + i] : (int8_t)0;
                sB[row * kPitch + 16 * chunk + i] = (okB && i < bytes_k) ? P.B[n * P.ldb + k + i] : (int8_t)0;
            }
        }
    }
}

template <int EPI>
__global__ void __launch_bounds__(256) gemm_tn_s8_kernel(GemmOperands P, GemmEpilogue E) {
    extern __shared__ __align__(16) int8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wm = warp & 1, wn = warp >> 1;  // 2 x 4 warps, each 64 x 32
    const int g = lane >> 2, tig = lane & 3;
    const int64_t mt = blockIdx.y, nt = blockIdx.x;
    const int64_t m0 = mt * kBM, n0 = nt * kBN;
    const int64_t nkb = s3r_cdiv(P.K, kBK);

    float accf[4][4][4];
    int32_t acci[4][4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int c = 0; c < 4; ++c) { accf[a][b][c] = 0.0f; acci[a][b][c] = 0; }

    load_stage(P, smem, smem + kBM * kPitch, m0, n0, 0);
    cp_async_commit();
    for (int64_t kb = 0; kb < nkb; ++kb) {
        int8_t* sA = smem + (kb & 1) * kStageBytes;
        int8_t* sB = sA + kBM * kPitch;
        if (kb + 1 < nkb) {
            int8_t* nA = smem + ((kb + 1) & 1) * kStageBytes;
            load_stage(P, nA, nA + kBM * kPitch, m0, n0, (kb + 1) * kBK);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
#pragma unroll
        for (int ks = 0; ks < kBK / 32; ++ks) {
            const int kc = ks * 32 + tig * 4;
            uint32_t af[4][4], bf[4][2];
#pragma unroll
            for (int mi = 0; mi < 4; ++mi) {
                const int r = wm * 64 + mi * 16 + g;
                af[mi][0] = *reinterpret_cast<const uint32_t*>(sA + r * kPitch + kc);
                af[mi][1] = *reinterpret_cast<const uint32_t*>(sA + (r + 8) * kPitch + kc);
                af[mi][2] = *reinterpret_cast<const uint32_t*>(sA + r * kPitch + kc + 16);
                af[mi][3] = *reinterpret_cast<const uint32_t*>(sA + (r + 8) * kPitch + kc + 16);
            }
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                const int r = wn * 32 + ni * 8 + g;
                bf[ni][0] = *reinterpret_cast<const uint32_t*>(sB + r * kPitch + kc);
                bf[ni][1] = *reinterpret_cast<const uint32_t*>(sB + r * kPitch + kc + 16);
            }
#pragma unroll
            for (int mi = 0; mi < 4; ++mi)
#pragma unroll
                for (int ni = 0; ni < 4; ++ni) mma_s8(acci[mi][ni], af[mi], bf[ni]);
        }
        if (EPI == kEpiDump) {
            const int64_t N = P.N;
#pragma unroll
            for (int mi = 0; mi < 4; ++mi)
#pragma unroll
                for (int ni = 0; ni < 4; ++ni)
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int64_t row = m0 + wm * 64 + mi * 16 + g + 8 * (r >> 1);
                        const int64_t col = n0 + wn * 32 + ni * 8 + tig * 2 + (r & 1);
                        if (row < P.M && col < N) E.dump[(row * N + col) * nkb + kb] = acci[mi][ni][r];
                        acci[mi][ni][r] = 0;
                    }
        } else {
            const float s = P.scale[mt * P.sm + nt * P.sn + kb * P.sk];
#pragma unroll
            for (int mi = 0; mi < 4; ++mi)
#pragma unroll
                for (int ni = 0; ni < 4; ++ni)
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        accf[mi][ni][r] = fmaf(s, (float)acci[mi][ni][r], accf[mi][ni][r]);
                        acci[mi][ni][r] = 0;
                    }
        }
        __syncthreads();
    }
    if (EPI == kEpiDump) return;

#pragma unroll
    for (int mi = 0; mi < 4; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int64_t row = m0 + wm * 64 + mi * 16 + g + 8 * (r >> 1);
                const int64_t col = n0 + wn * 32 + ni * 8 + tig * 2 + (r & 1);
                if (row >= P.M || col >= P.N) continue;
                float out = accf[mi][ni][r];
                if (EPI == kEpiDX) {
                    if (E.ec_mode != S3R_EC_NONE)
                        out = out - fmaf(E.eps[row], (float)E.rowsum[col], E.v[(row / E.S) * P.N + col]);
                    if (E.s_x) out = out / E.s_x[row];
                    float* dst = E.C + row * E.ldc + col;
                    if (E.accumulate) out = out + *dst;
                    *dst = out;
                } else {
                    if (E.ec_mode == S3R_EC_TWO_WAY) {
                        float corr = E.p[row];
                        for (int64_t b = 0; b < E.B; ++b)
                            corr = fmaf((float)E.xsum[b * P.M + row], E.colmean[b * P.N + col] - E.mu[b], corr);
                        out = out - corr;
                    }
                    if (E.s_w) out = out / E.s_w[col];
                    E.C[row * E.ldc + col] = out;
                }
            }
}

// dst[c, r] = src[r, c] for an int8 [R, C] matrix; dst row stride ldd.
__global__ void __launch_bounds__(256) transpose_s8_kernel(const int8_t* src, int64_t R, int64_t C, int64_t lds,
                                                           int8_t* dst, int64_t ldd) {
    __shared__ int8_t tile[64][65];
    const int64_t r0 = (int64_t)blockIdx.y * 64, c0 = (int64_t)blockIdx.x * 64;
    const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;  // 64 x 4
    for (int i = ty; i < 64; i += 4) {
        const int64_t r = r0 + i, c = c0 + tx;
        tile[i][tx] = (r < R && c < C) ? src[r * lds + c] : (int8_t)0;
    }
    __syncthreads();
    for (int i = ty; i < 64; i += 4) {
        const int64_t c = c0 + i, r = r0 + tx;
        if (c < C && r < R) dst[c * ldd + r] = tile[tx][i];
    }
}

}  // namespace s3r

using namespace s3r;

// tcgen05 path for fp16-carried codes (gemm_umma.cu)
int umma_gemm_dx(const void* Q, const float* tile_scale, const void* W, int64_t T, int64_t N, int64_t K,
                 const float* s_x, int ec_mode, const float* eps, const int32_t* rowsum, const float* v, int64_t S,
                 float* dX, int accumulate, int32_t* dump, int* d_status, cudaStream_t stream);
int umma_gemm_dx2(const void* Q, const float* tile_scale, const void* W, const float* eps, const int32_t* rowsum,
                  const float* v, const void* Q3, const float* tile_scale3, const void* W3, const float* eps3,
                  const int32_t* rowsum3, const float* v3, int64_t T, int64_t N, int64_t K, const float* s_x,
                  int ec_mode, int64_t S, float* dX, int accumulate, int32_t* dump, int* d_status,
                  cudaStream_t stream);
int umma_gemm_dw(const void* X, const void* Q, const float* tile_scale, int64_t T, int64_t K, int64_t N,
                 const float* s_w, int ec_mode, const float* colmean, const float* mu, const int32_t* xsum,
                 const float* p, int64_t S, float* dW, int32_t* dump, int* d_status, cudaStream_t stream);

static int ensure_gemm_smem() {
    const char* what = "mma.sync gemm: cudaFuncSetAttribute";
    int st = s3r_kernel_smem((const void*)gemm_tn_s8_kernel<kEpiDX>, kGemmSmem, what);
    if (!st) st = s3r_kernel_smem((const void*)gemm_tn_s8_kernel<kEpiDW>, kGemmSmem, what);
    if (!st) st = s3r_kernel_smem((const void*)gemm_tn_s8_kernel<kEpiDump>, kGemmSmem, what);
    return st;
}

template <int EPI>
static int launch_gemm(const GemmOperands& P, const GemmEpilogue& E, cudaStream_t stream) {
    int st = ensure_gemm_smem();
    if (st) return st;
    if (s3r_cdiv(P.M, kBM) > 65535) return S3R_ERR_UNSUPPORTED;
    dim3 grid((unsigned)s3r_cdiv(P.N, kBN), (unsigned)s3r_cdiv(P.M, kBM));
    gemm_tn_s8_kernel<EPI><<<grid, 256, kGemmSmem, stream>>>(P, E);
    S3R_CHECK_LAUNCH();
    return S3R_OK;
}

static int64_t pad16(int64_t x) { return (x + 15) / 16 * 16; }

extern "C" size_t int8_gemm_dw_workspace_size(int64_t T, int64_t K, int64_t N, int code_format) {
    if (T <= 0 || K <= 0 || N <= 0 || code_format != S3R_CODES_S8) return 0;
    return (size_t)(K + N) * (size_t)pad16(T) + 512;
}

static int transpose_pair(const int8_t* X8, const int8_t* Q, int64_t T, int64_t K, int64_t N, void* ws,
                          size_t ws_bytes, int8_t** Xt, int8_t** Qt, cudaStream_t stream) {
    if (!ws || ws_bytes < int8_gemm_dw_workspace_size(T, K, N, S3R_CODES_S8)) return S3R_ERR_WORKSPACE;
    const int64_t ldt = pad16(T);
    uintptr_t base = ((uintptr_t)ws + 255) & ~(uintptr_t)255;
    *Xt = reinterpret_cast<int8_t*>(base);
    *Qt = *Xt + K * ldt;
    transpose_s8_kernel<<<dim3((unsigned)s3r_cdiv(K, 64), (unsigned)s3r_cdiv(T, 64)), 256, 0, stream>>>(X8, T, K, K,
                                                                                                     *Xt, ldt);
    S3R_CHECK_LAUNCH();
    transpose_s8_kernel<<<dim3((unsigned)s3r_cdiv(N, 64), (unsigned)s3r_cdiv(T, 64)), 256, 0, stream>>>(Q, T, N, N,
                                                                                                     *Qt, ldt);
    S3R_CHECK_LAUNCH();
    return S3R_OK;
}

extern "C" int int8_gemm_dx(const void* Qv, const float* tile_scale, const void* W8v, int code_format, int64_t T,
                            int64_t N, int64_t K, const float* s_x, int ec_mode, const float* eps,
                            const int32_t* rowsum, const float* v, int64_t S, float* dX, int accumulate, int* d_status,
                            cudaStream_t stream) {
    if (T < 0 || N < 0 || K < 0) return S3R_ERR_ARG;
    if (code_format != S3R_CODES_S8 && code_format != S3R_CODES_F16) return S3R_ERR_ARG;
    if (T == 0 || K == 0) return S3R_OK;
    if (!Qv || !tile_scale || !W8v || !dX) return S3R_ERR_ARG;
    if (ec_mode < S3R_EC_NONE || ec_mode > S3R_EC_DW_ONLY) return S3R_ERR_ARG;
    if (ec_mode == S3R_EC_DW_ONLY) ec_mode = S3R_EC_NONE;   // the ablation corrects dW only
    if (ec_mode != S3R_EC_NONE && (!eps || !rowsum || !v || S <= 0 || T % S != 0)) return S3R_ERR_ARG;
    if (N == 0) return S3R_ERR_SHAPE;
    if (code_format == S3R_CODES_F16)
        return umma_gemm_dx(Qv, tile_scale, W8v, T, N, K, s_x, ec_mode, eps, rowsum, v, S > 0 ? S : T, dX,
                            accumulate, nullptr, d_status, stream);
    const int8_t* Q = static_cast<const int8_t*>(Qv);
    const int8_t* W8 = static_cast<const int8_t*>(W8v);
    const bool aligned = s3r_aligned16(Q) && s3r_aligned16(W8) && N % 16 == 0;
    GemmOperands P{Q, N, W8, N, T, K, N, tile_scale, s3r_cdiv(N, kTile), 0, 1, aligned};
    GemmEpilogue E{};
    E.C = dX; E.ldc = K; E.s_x = s_x; E.eps = eps; E.rowsum = rowsum; E.v = v; E.accumulate = accumulate;
    E.ec_mode = ec_mode; E.S = S > 0 ? S : T;
    return launch_gemm<kEpiDX>(P, E, stream);
}

extern "C" int int8_gemm_dx_sum(const struct s3r_dx_term* terms, int n_terms, int code_format, int64_t T,
                                int64_t N, int64_t K, const float* s_x, int ec_mode, int64_t S, float* dX,
                                int accumulate, int* d_status, cudaStream_t stream) {
    if (!terms || n_terms < 1 || n_terms > S3R_DX_MAX_TERMS) return S3R_ERR_ARG;
    if (T < 0 || N < 0 || K < 0) return S3R_ERR_ARG;
    if (code_format != S3R_CODES_S8 && code_format != S3R_CODES_F16) return S3R_ERR_ARG;
    if (T == 0 || K == 0) return S3R_OK;
    if (!dX) return S3R_ERR_ARG;
    if (ec_mode < S3R_EC_NONE || ec_mode > S3R_EC_DW_ONLY) return S3R_ERR_ARG;
    if (ec_mode == S3R_EC_DW_ONLY) ec_mode = S3R_EC_NONE;   // the ablation corrects dW only
    for (int i = 0; i < n_terms; ++i) {
        const s3r_dx_term& t = terms[i];
        if (!t.Q || !t.tile_scale || !t.W8) return S3R_ERR_ARG;
        if (ec_mode != S3R_EC_NONE && (!t.eps || !t.rowsum || !t.v || S <= 0 || T % S != 0)) return S3R_ERR_ARG;
    }
    if (N == 0) return S3R_ERR_SHAPE;
    if (code_format == S3R_CODES_F16) {
        const s3r_dx_term& a = terms[0];
        const s3r_dx_term* b = n_terms > 1 ? &terms[1] : nullptr;
        return umma_gemm_dx2(a.Q, a.tile_scale, a.W8, a.eps, a.rowsum, a.v, b ? b->Q : nullptr,
                             b ? b->tile_scale : nullptr, b ? b->W8 : nullptr, b ? b->eps : nullptr,
                             b ? b->rowsum : nullptr, b ? b->v : nullptr, T, N, K, s_x, ec_mode, S > 0 ? S : T, dX,
                             accumulate, nullptr, d_status, stream);
    }
    // the warp-level path runs one launch per term, the later ones accumulating
    for (int i = 0; i < n_terms; ++i) {
        const s3r_dx_term& t = terms[i];
        int st = int8_gemm_dx(t.Q, t.tile_scale, t.W8, code_format, T, N, K, s_x, ec_mode, t.eps, t.rowsum, t.v, S,
                              dX, i > 0 ? 1 : accumulate, d_status, stream);
        if (st) return st;
    }
    return S3R_OK;
}

extern "C" int int8_gemm_dw(const void* X8v, const void* Qv, const float* tile_scale, int code_format, int64_t T,
                            int64_t K, int64_t N, const float* s_w, int ec_mode, const float* colmean, const float* mu,
                            const int32_t* xsum, const float* p, int64_t S, float* dW, void* workspace,
                            size_t workspace_bytes, int* d_status, cudaStream_t stream) {
    if (T < 0 || N < 0 || K < 0) return S3R_ERR_ARG;
    if (code_format != S3R_CODES_S8 && code_format != S3R_CODES_F16) return S3R_ERR_ARG;
    if (K == 0 || N == 0) return S3R_OK;
    if (!X8v || !Qv || !tile_scale || !dW) return S3R_ERR_ARG;
    if (ec_mode < S3R_EC_NONE || ec_mode > S3R_EC_DW_ONLY) return S3R_ERR_ARG;
    if (ec_mode == S3R_EC_DW_ONLY) ec_mode = S3R_EC_TWO_WAY;   // dW carries the whole correction
    if (ec_mode == S3R_EC_TWO_WAY && (!colmean || !mu || !xsum || !p || S <= 0 || T % S != 0)) return S3R_ERR_ARG;
    if (T == 0) return S3R_ERR_SHAPE;
    if (code_format == S3R_CODES_F16)
        return umma_gemm_dw(X8v, Qv, tile_scale, T, K, N, s_w, ec_mode, colmean, mu, xsum, p, S > 0 ? S : T, dW,
                            nullptr, d_status, stream);
    const int8_t* X8 = static_cast<const int8_t*>(X8v);
    const int8_t* Q = static_cast<const int8_t*>(Qv);
    int8_t *Xt, *Qt;
    int st = transpose_pair(X8, Q, T, K, N, workspace, workspace_bytes, &Xt, &Qt, stream);
    if (st) return st;
    const int64_t ldt = pad16(T);
    GemmOperands P{Xt, ldt, Qt, ldt, K, N, T, tile_scale, 0, 1, s3r_cdiv(N, kTile), true};
    GemmEpilogue E{};
    E.C = dW; E.ldc = N; E.s_w = s_w; E.colmean = colmean; E.mu = mu; E.xsum = xsum; E.p = p;
    E.ec_mode = ec_mode; E.S = S > 0 ? S : T; E.B = (S > 0) ? T / S : 1;
    return launch_gemm<kEpiDW>(P, E, stream);
}

extern "C" int s3r_debug_dx_blocks(const void* Qv, const void* W8v, int code_format, int64_t T, int64_t N,
                                   int64_t K, int32_t* out_dx, cudaStream_t stream) {
    if (T <= 0 || N <= 0 || K <= 0 || !Qv || !W8v || !out_dx) return S3R_ERR_ARG;
    if (code_format == S3R_CODES_F16)
        return umma_gemm_dx(Qv, nullptr, W8v, T, N, K, nullptr, 0, nullptr, nullptr, nullptr, T, nullptr, 0, out_dx,
                            nullptr, stream);
    if (code_format != S3R_CODES_S8) return S3R_ERR_ARG;
    const int8_t* Q = static_cast<const int8_t*>(Qv);
    const int8_t* W8 = static_cast<const int8_t*>(W8v);
    const bool aligned = s3r_aligned16(Q) && s3r_aligned16(W8) && N % 16 == 0;
    GemmOperands P{Q, N, W8, N, T, K, N, nullptr, 0, 0, 0, aligned};
    GemmEpilogue E{};
    E.dump = out_dx;
    return launch_gemm<kEpiDump>(P, E, stream);
}

extern "C" int s3r_debug_dw_blocks(const void* X8v, const void* Qv, int code_format, int64_t T, int64_t K, int64_t N,
                                   int32_t* out_dw, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (T <= 0 || N <= 0 || K <= 0 || !X8v || !Qv || !out_dw) return S3R_ERR_ARG;
    if (code_format == S3R_CODES_F16)
        return umma_gemm_dw(X8v, Qv, nullptr, T, K, N, nullptr, 0, nullptr, nullptr, nullptr, nullptr, T, nullptr,
                            out_dw, nullptr, stream);
    if (code_format != S3R_CODES_S8) return S3R_ERR_ARG;
    const int8_t* X8 = static_cast<const int8_t*>(X8v);
    const int8_t* Q = static_cast<const int8_t*>(Qv);
    int8_t *Xt, *Qt;
    int st = transpose_pair(X8, Q, T, K, N, workspace, workspace_bytes, &Xt, &Qt, stream);
    if (st) return st;
    const int64_t ldt = pad16(T);
    GemmOperands P{Xt, ldt, Qt, ldt, K, N, T, nullptr, 0, 0, 0, true};
    GemmEpilogue E{};
    E.dump = out_dw;
    return launch_gemm<kEpiDump>(P, E, stream);
}
