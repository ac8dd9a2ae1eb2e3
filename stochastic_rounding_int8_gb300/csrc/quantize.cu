// quantize.cu -- tile quantizers of the backward gradient (S3R, independent SR,
// RTNE), the SwiGLU-fused variant and the forward-operand RTNE kernels.
//
// Paper: "Efficient Quantization Training with Stochastic Rounding via
// Structured Subspace Randomness" §III-A (fold, per-tensor/tile step, SR
// operator), §III-B (one threshold per token broadcast over the hidden
// dimension; one quantized tensor for both products), §IV-B (baselines).
//
// Design (HBM-bound): one CTA owns one 128x128 tile.  Every thread holds a
// 16-byte chunk (8 columns) of RPT rows in registers, loaded once with 128-bit
// coalesced loads; the tile absmax is a warp redux.sync on the IEEE bit
// patterns (which also flags NaN/Inf) then a CTA reduction; the per-token
// Philox threshold is computed by one lane per row and broadcast with
// __shfl_sync; codes are written once as 8-byte stores; the error partials are
// reduced with shuffles and a small shared-memory pass, in a fixed order.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdio>

#include "common.cuh"

namespace s3r {

enum QMode { kRTNE = 0, kS3R = 1, kINDEP = 2, kS3R7 = 3, kBCAST = 4 };

// Modes with one threshold per row of the tensor (shared by its channels), one
// threshold tensor for both products, and the S3R-EC error partials.
__host__ __device__ constexpr bool row_mode(int m) { return m == kS3R || m == kS3R7 || m == kBCAST; }

// Per-thread geometry of a 128x128 tile: chunk c (8 columns), rows r0 + j*RSTRIDE.
template <int RPT>
struct TileGeom {
    static constexpr int kThreads = 16 * (128 / RPT);
    static constexpr int kRowStride = 128 / RPT;
    static constexpr int kWarps = kThreads / 32;
};

struct QuantOut {
    void* Q;
    int fmt;  // S3R_CODES_S8 or S3R_CODES_F16
    float* scale;
    float* tok;
    float* col;
    uint32_t tensor_id;
};

struct QuantCommon {
    int64_t T, N;
    int64_t ntc;
    uint32_t seed_lo;
    int* d_status;
    bool vec_store;  // Q rows aligned for one vector store per 8-code chunk
    int64_t S;       // tokens per example (Phi_bcast); 0: one example
    const uint32_t* tensor_amax;   // per-tensor step: bits of max |g| over the tensor (null: per tile)
};

// The threshold of row t under a row-threshold mode.
template <int MODE>
__device__ __forceinline__ float row_threshold(uint64_t t, const QuantCommon& C, uint32_t tensor_id) {
    if (MODE == kS3R7) return token_threshold7(t, C.seed_lo, tensor_id);
    if (MODE == kBCAST) return example_threshold(C.S > 0 ? t / (uint64_t)C.S : 0u, C.seed_lo, tensor_id);
    return token_threshold(t, C.seed_lo, tensor_id);
}

// Block-wide max of non-negative float bit patterns (NaN/Inf compare largest).
template <int WARPS>
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t* smem) {
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) smem[warp] = v;
    __syncthreads();
    uint32_t m = 0;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) m = max(m, smem[w]);
    __syncthreads();
    return m;
}

// Round one thread's folded values to codes, write them, and accumulate the
// tile's error partials.  ng holds the folded gradient NEGATED (-g), so the
// error e = delta*q - g is a single fma(delta, q, ng).  amax_bits is the tile
// absmax.  inv = 127/amax rounded toward zero keeps |y| <= 127, so no code can
// leave [-127, 127] and no clamp is needed.
template <int MODE, int RPT, int FMT = -1>
__device__ __forceinline__ void round_and_store(const float (&ng)[RPT][8], uint32_t amax_bits, int64_t t0, int64_t n0,
                                                int r0, int c, const QuantCommon& C, const QuantOut& O,
                                                float* col_smem /* [WARPS][128] */) {
    using Geo = TileGeom<RPT>;
    const int fmt = FMT >= 0 ? FMT : O.fmt;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t nc0 = n0 + 8 * c;
    const bool nonfinite = amax_bits >= 0x7F800000u;   // uniform across the CTA
    const float amax = __uint_as_float(amax_bits);
    const float d = nonfinite ? __uint_as_float(0x7FC00000u) : amax / 127.0f;
    const float inv = (amax_bits == 0u || nonfinite) ? 0.0f : __fdiv_rz(127.0f, amax);
    if (threadIdx.x == 0) {
        O.scale[(t0 / kTile) * C.ntc + (n0 / kTile)] = d;
        if (nonfinite) set_status(C.d_status, S3R_ERR_NONFINITE);
    }

    // thresholds of my rows: lane (half*16 + j) draws the one of row r0 + j*RSTRIDE
    float u_row[RPT];
    if (row_mode(MODE)) {
        float mine = 0.0f;
        if (c < RPT) mine = row_threshold<MODE>((uint64_t)(t0 + r0 + c * Geo::kRowStride), C, O.tensor_id);
#pragma unroll
        for (int j = 0; j < RPT; ++j) u_row[j] = __shfl_sync(0xFFFFFFFFu, mine, (lane & 16) + j);
    }

    const float2 ninv2 = make_float2(-inv, -inv), d2 = make_float2(d, d);
    float2 colsum[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) colsum[k] = make_float2(0.0f, 0.0f);

#pragma unroll
    for (int j = 0; j < RPT; ++j) {
        const int64_t t = t0 + r0 + j * Geo::kRowStride;
        float u8[8];
        if (MODE == kINDEP) {
            if ((C.N & 3) == 0) {
                const uint64_t e0 = (uint64_t)t * (uint64_t)C.N + (uint64_t)nc0;  // multiple of 4
                const uint64_t ctr = e0 >> 2;
                const Philox4 a = philox4x32_10((uint32_t)ctr, (uint32_t)(ctr >> 32), 0u, 0u, C.seed_lo, O.tensor_id);
                const Philox4 b =
                    philox4x32_10((uint32_t)(ctr + 1), (uint32_t)((ctr + 1) >> 32), 0u, 0u, C.seed_lo, O.tensor_id);
                u8[0] = unit24(a.x); u8[1] = unit24(a.y); u8[2] = unit24(a.z); u8[3] = unit24(a.w);
                u8[4] = unit24(b.x); u8[5] = unit24(b.y); u8[6] = unit24(b.z); u8[7] = unit24(b.w);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint64_t e = (uint64_t)t * (uint64_t)C.N + (uint64_t)(nc0 + i);
                    const uint64_t ctr = e >> 2;
                    const Philox4 a = philox4x32_10((uint32_t)ctr, (uint32_t)(ctr >> 32), 0u, 0u, C.seed_lo, O.tensor_id);
                    const uint32_t w = (e & 3) == 0 ? a.x : (e & 3) == 1 ? a.y : (e & 3) == 2 ? a.z : a.w;
                    u8[i] = unit24(w);
                }
            }
        }
        // qm = kMagic + q (exact): floor and round-to-nearest are adds of kMagic
        // on the FMA pipe, and the int8 code is the low byte of qm's bits
        float qv[8], qm[8];
        float2 rs = make_float2(0.0f, 0.0f);
        const float2 M2 = make_float2(kMagic, kMagic);
        if (!nonfinite) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 g2 = make_float2(ng[j][2 * k], ng[j][2 * k + 1]);
                const float2 y = f2_mul(g2, ninv2);                  // = g * inv, |y| <= 127
                float2 m;
                if (MODE == kRTNE) {
                    // per lane: a packed add that is the product's only use would be fused into an fma
                    m = make_float2(__fadd_rn(y.x, kMagic), __fadd_rn(y.y, kMagic));   // kMagic + rint(y)
                } else {
                    const float2 fm = f2_add_rm(y, M2);              // kMagic + floor(y)
                    const float2 f = f2_sub(fm, M2);                 // floor(y), exact
                    const float2 p = f2_sub(y, f);                   // residual in [0, 1), exact
                    const float ua = row_mode(MODE) ? u_row[j] : u8[2 * k];
                    const float ub = row_mode(MODE) ? u_row[j] : u8[2 * k + 1];
                    m = f2_add(fm, make_float2(lt_one(ua, p.x), lt_one(ub, p.y)));   // + [u < p]
                }
                const float2 q = f2_sub(m, M2);                      // the code, exact
                qm[2 * k] = m.x;
                qm[2 * k + 1] = m.y;
                qv[2 * k] = q.x;
                qv[2 * k + 1] = q.y;
                const float2 e = f2_fma(d2, q, g2);                  // delta*q - g
                rs = f2_add(rs, e);
                colsum[k] = f2_add(colsum[k], e);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                qv[i] = 0.0f;
                qm[i] = kMagic;
            }
        }
        const float rowsum = rs.x + rs.y;
        if (t < C.T) {
            if (fmt == S3R_CODES_S8) {
                uint32_t w[2];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const uint32_t a = __float_as_uint(qm[4 * k]), b = __float_as_uint(qm[4 * k + 1]);
                    const uint32_t cc = __float_as_uint(qm[4 * k + 2]), dd = __float_as_uint(qm[4 * k + 3]);
                    w[k] = __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(cc, dd, 0x0040), 0x5410);
                }
                int8_t* dst = static_cast<int8_t*>(O.Q) + t * C.N + nc0;
                if (C.vec_store && nc0 + 8 <= C.N) {
                    *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (nc0 + i < C.N) dst[i] = (int8_t)__float2int_rn(qv[i]);
                }
            } else {
                // the same integer in an IEEE half (exact for |q| <= 2048)
                uint32_t hw[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const __half2 h2 = __floats2half2_rn(qv[2 * k], qv[2 * k + 1]);
                    hw[k] = *reinterpret_cast<const uint32_t*>(&h2);
                }
                __half* dst = static_cast<__half*>(O.Q) + t * C.N + nc0;
                if (C.vec_store && nc0 + 8 <= C.N) {
                    *reinterpret_cast<uint4*>(dst) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (nc0 + i < C.N) dst[i] = __float2half_rn(qv[i]);
                }
            }
        }
        if (O.tok) {
            float r = rowsum;
            r += __shfl_xor_sync(0xFFFFFFFFu, r, 8);
            r += __shfl_xor_sync(0xFFFFFFFFu, r, 4);
            r += __shfl_xor_sync(0xFFFFFFFFu, r, 2);
            r += __shfl_xor_sync(0xFFFFFFFFu, r, 1);
            if (c == 0 && t < C.T) O.tok[t * C.ntc + n0 / kTile] = r;
        }
    }
    if (O.col) {
        float cs[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            cs[2 * k] = colsum[k].x + __shfl_xor_sync(0xFFFFFFFFu, colsum[k].x, 16);
            cs[2 * k + 1] = colsum[k].y + __shfl_xor_sync(0xFFFFFFFFu, colsum[k].y, 16);
        }
        if (lane < 16) {
#pragma unroll
            for (int i = 0; i < 8; ++i) col_smem[warp * 128 + 8 * c + i] = cs[i];
        }
        __syncthreads();
        if (threadIdx.x < 128) {
            float sum = 0.0f;
#pragma unroll
            for (int w = 0; w < Geo::kWarps; ++w) sum += col_smem[w * 128 + threadIdx.x];
            if (n0 + threadIdx.x < C.N) O.col[(t0 / kTile) * C.N + n0 + threadIdx.x] = sum;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Backward-gradient tile quantizer: bf16 G -> fold -> tile scale -> codes.
// ---------------------------------------------------------------------------
struct TileQuantArgs {
    const uint16_t* G;
    int64_t ldg;
    const float* s_x;
    const float* s_w;
    bool vec_load;  // rows 16-byte aligned
};

template <int MODE>
__global__ void __launch_bounds__(256) quantize_tile_kernel(TileQuantArgs A, QuantCommon C, QuantOut O) {
    constexpr int RPT = 8;
    using Geo = TileGeom<RPT>;
    __shared__ uint32_t red[Geo::kWarps];
    __shared__ float col_smem[Geo::kWarps * 128];
    const int c = threadIdx.x & 15, r0 = threadIdx.x >> 4;
    const int64_t t0 = (int64_t)blockIdx.y * kTile, n0 = (int64_t)blockIdx.x * kTile;
    const int64_t nc0 = n0 + 8 * c;

    uint4 raw[RPT];
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
        const int64_t t = t0 + r0 + j * Geo::kRowStride;
        raw[j] = make_uint4(0u, 0u, 0u, 0u);
        if (t < C.T) {
            const uint16_t* src = A.G + t * A.ldg + nc0;
            if (A.vec_load && nc0 + 8 <= C.N) {
                raw[j] = __ldg(reinterpret_cast<const uint4*>(src));
            } else {
                uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (nc0 + i < C.N) w[i >> 1] |= (uint32_t)src[i] << (16 * (i & 1));
                raw[j] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    }
    float sw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) sw[i] = (A.s_w && nc0 + i < C.N) ? __ldg(A.s_w + nc0 + i) : 1.0f;

    float g[RPT][8];
    uint32_t amax_bits = 0u;
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
        const int64_t t = t0 + r0 + j * Geo::kRowStride;
        // negated fold: (-s_x) * G * s_w == -((s_x * G) * s_w) exactly
        const float nsx = (A.s_x && t < C.T) ? -__ldg(A.s_x + t) : -1.0f;
        const uint32_t w[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float v = (i & 1) ? bf16_hi(w[i >> 1]) : bf16_lo(w[i >> 1]);
            v = nsx * v;
            if (A.s_w) v = v * sw[i];
            g[j][i] = v;
            amax_bits = max(amax_bits, __float_as_uint(v) & 0x7FFFFFFFu);
        }
    }
    amax_bits = block_max_u32<Geo::kWarps>(amax_bits, red);
    if (C.tensor_amax) amax_bits = __ldg(C.tensor_amax);   // one step for the whole tensor
    round_and_store<MODE, RPT>(g, amax_bits, t0, n0, r0, c, C, O, col_smem);
}

// ---------------------------------------------------------------------------
// Persistent variant: each CTA walks tiles tile = blockIdx.x + i * gridDim.x;
// a TMA engine copies the next 128x128 bf16 tile into the other half of a
// two-buffer shared-memory ring while the current one is rounded, so the HBM
// stream never waits for the arithmetic.  The folded values stay in registers
// after the absmax pass, which frees the buffer for the next copy early.
// ---------------------------------------------------------------------------
constexpr uint64_t kQuantWaitNs = 2000000000ull;

__device__ __forceinline__ uint64_t q_gtime() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ bool q_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns = kQuantWaitNs) {
    uint32_t ok = 0;
    const uint64_t t0 = q_gtime();
    while (true) {
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
        if (q_gtime() - t0 > limit_ns) return false;
    }
}

// Test hook: q_wait on a barrier that nothing arrives on, with a short limit;
// the waiter records how long it waited and sets S3R_ERR_TIMEOUT.
__global__ void __launch_bounds__(32) q_wait_probe_kernel(uint64_t limit_ns, int* d_status,
                                                          unsigned long long* waited_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = (uint32_t)__cvta_generic_to_shared(&bar);
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        const uint64_t t0 = q_gtime();
        const bool ok = q_wait(b, 0u, limit_ns);
        *waited_ns = q_gtime() - t0;
        if (!ok) set_status(d_status, S3R_ERR_TIMEOUT);
    }
}
__device__ __forceinline__ void q_issue_tile(uint32_t dst, const CUtensorMap* map, int32_t col, int32_t row,
                                             uint32_t bar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(kTile * kTile * 2)
                 : "memory");
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"((uint64_t)map), "r"(col), "r"(row), "r"(bar)
        : "memory");
}

// Round RPT rows of 8 values (rows RS apart; gpair(j, q) gives values 2q and
// 2q + 1 of row j) to codes and store them; with
// ERR, add -e = g - delta*q (one rounding: the exact negation of delta*q - g)
// into the row sums and the per-column sums.
//   SR: q = floor(y) + [u < frac(y)] = ceil(y - u) for u in [0, 1).  y - u
//   rounded up never passes an integer, so its ceiling is exact, and adding
//   kMagic rounded up takes it: m = kMagic + q, exact.  RTNE: m = kMagic + y
//   rounded to nearest.  The int8 code is the low byte of m's bits.
// q0 points at my first row's 8 codes; rows_left: row j is stored iff RS j < rows_left.
// The codes are stored as streaming writes (evict first): the next reader is a
// GEMM several launches later, and keeping them out of L2 leaves it to the
// gradient being read (fp16 codes on [16384, 8192]: 106 -> 102 us).
template <int MODE, int FMT, int RPT, int RS, bool ERR, typename PairFn>
__device__ __forceinline__ void round_rows(PairFn gpair, float d, float inv, bool nonfinite, const float* u0,
                                           int u_step, void* q0, int64_t row_step, int rows_left, int64_t t_first,
                                           int nc0, int64_t N, uint32_t seed_lo, uint32_t tensor_id,
                                           float (&rsum)[RPT], float2 (&colsum)[4]) {
    const float2 M2 = make_float2(kMagic, kMagic), inv2 = make_float2(inv, inv), nd2 = make_float2(-d, -d);
#pragma unroll
    for (int q = 0; q < 4; ++q) colsum[q] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
        float u8[8];
        if (MODE == kINDEP) {
            const int64_t t = t_first + RS * j;
            if ((N & 3) == 0) {
                const uint64_t ctr = ((uint64_t)t * (uint64_t)N + (uint64_t)nc0) >> 2;
                const Philox4 a = philox4x32_10((uint32_t)ctr, (uint32_t)(ctr >> 32), 0u, 0u, seed_lo, tensor_id);
                const Philox4 b =
                    philox4x32_10((uint32_t)(ctr + 1), (uint32_t)((ctr + 1) >> 32), 0u, 0u, seed_lo, tensor_id);
                u8[0] = unit24(a.x); u8[1] = unit24(a.y); u8[2] = unit24(a.z); u8[3] = unit24(a.w);
                u8[4] = unit24(b.x); u8[5] = unit24(b.y); u8[6] = unit24(b.z); u8[7] = unit24(b.w);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint64_t e = (uint64_t)t * (uint64_t)N + (uint64_t)(nc0 + i);
                    const uint64_t ctr = e >> 2;
                    const Philox4 a = philox4x32_10((uint32_t)ctr, (uint32_t)(ctr >> 32), 0u, 0u, seed_lo, tensor_id);
                    const uint32_t w = (e & 3) == 0 ? a.x : (e & 3) == 1 ? a.y : (e & 3) == 2 ? a.z : a.w;
                    u8[i] = unit24(w);
                }
            }
        }
        const float ut = row_mode(MODE) ? u0[j * u_step] : 0.0f;
        float qv[8], qm[8];
        float2 rs = make_float2(0.0f, 0.0f);
        if (!nonfinite) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 g2 = gpair(j, q);   // values 8 c + 2 q, 8 c + 2 q + 1 of row j
                const float2 y = f2_mul(g2, inv2);   // |y| <= 127
                float2 m;
                if (MODE == kRTNE) {
                    // per lane: a packed add that is the product's only use would be fused into an fma
                    m = make_float2(__fadd_rn(y.x, kMagic), __fadd_rn(y.y, kMagic));
                } else {
                    const float2 uu = row_mode(MODE) ? make_float2(ut, ut) : make_float2(u8[2 * q], u8[2 * q + 1]);
                    m = f2_add_rp(f2_sub_rp(y, uu), M2);
                }
                const float2 qq = f2_sub(m, M2);   // the code, exact
                qm[2 * q] = m.x;
                qm[2 * q + 1] = m.y;
                qv[2 * q] = qq.x;
                qv[2 * q + 1] = qq.y;
                if (ERR) {
                    const float2 ne = f2_fma(nd2, qq, g2);   // g - delta*q = -e
                    rs = f2_add(rs, ne);
                    colsum[q] = f2_add(colsum[q], ne);
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                qv[i] = 0.0f;
                qm[i] = kMagic;
            }
        }
        rsum[j] = rs.x + rs.y;
        if (RS * j < rows_left) {
            if (FMT == 0) {
                uint32_t w[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t a = __float_as_uint(qm[4 * h]), b = __float_as_uint(qm[4 * h + 1]);
                    const uint32_t cc = __float_as_uint(qm[4 * h + 2]), dd = __float_as_uint(qm[4 * h + 3]);
                    w[h] = __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(cc, dd, 0x0040), 0x5410);
                }
                int8_t* dst = static_cast<int8_t*>(q0) + j * row_step;
                if (nc0 + 8 <= N) {
                    __stcs(reinterpret_cast<uint2*>(dst), make_uint2(w[0], w[1]));   // streaming: evict first
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (nc0 + i < N) dst[i] = (int8_t)__float2int_rn(qv[i]);
                }
            } else {
                // the same integer in an IEEE half (exact for |q| <= 2048)
                uint32_t hw[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const __half2 h2 = __floats2half2_rn(qv[2 * q], qv[2 * q + 1]);
                    hw[q] = *reinterpret_cast<const uint32_t*>(&h2);
                }
                __half* dst = static_cast<__half*>(q0) + j * row_step;
                if (nc0 + 8 <= N) {
                    __stcs(reinterpret_cast<uint4*>(dst), make_uint4(hw[0], hw[1], hw[2], hw[3]));   // streaming: evict first
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (nc0 + i < N) dst[i] = __float2half_rn(qv[i]);
                }
            }
        }
    }
}

// 16 lanes (c = lane & 15) of a row group hold RPT row sums each: a
// reduce-scatter (halving exchanges, then plain ones) leaves lane c with the
// full sum of row c / (16 / RPT), in a fixed order.
template <int RPT>
__device__ __forceinline__ float scatter_rows16(const float (&v)[RPT], int c) {
    float a[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) a[i] = v[i];
    int n = RPT;
#pragma unroll
    for (int x = 8; x >= 1; x >>= 1) {
        if (n > 1) {
            const int h = n / 2;
            const bool hi = c & x;
#pragma unroll
            for (int i = 0; i < RPT / 2; ++i) {
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

// Persistent quantizer.  CTA b owns the contiguous tile range
// [b ntiles / grid, (b + 1) ntiles / grid) in row-major tile order, so its
// consecutive tiles mostly share a row block and reuse that block's
// thresholds.  A TMA engine keeps up to kQStages 128 x 128 bf16 tiles in
// flight in a shared-memory ring.  The side data of a tile -- the row scales
// with the row thresholds, and the column scales -- is fetched two tiles
// ahead (threads 0..127 own a row, 128..255 a column) into a three-slot ring.
// One CTA barrier per tile: every thread waits for the tile's copy itself;
// the barrier after the absmax hands the stage back to the TMA engine, makes
// the warps' maxima visible, and also orders the exchanges around it -- the
// previous tile's column sums (double-buffered) are added after it, and the
// side-data slot that the previous tile used is refilled after it.
constexpr int kQStages = 3;
constexpr int kQTileBytes = kTile * kTile * 2;
constexpr int kQuantTmaSmem = kQStages * kQTileBytes + 8 * kQStages;

// side data of the tile in row block rb, column block cb for this thread:
// (row scale, threshold) or (column scale, 0)
template <int MODE>
__device__ __forceinline__ float2 q_side(const TileQuantArgs& A, const QuantCommon& C, uint32_t tensor_id, int rb,
                                         int cb, float& u_mine, int& u_rb) {
    if (threadIdx.x < kTile) {
        const int64_t t = (int64_t)rb * kTile + threadIdx.x;
        const float sx = (A.s_x && t < C.T) ? __ldg(A.s_x + t) : 1.0f;
        if (row_mode(MODE) && rb != u_rb) {
            u_mine = row_threshold<MODE>((uint64_t)t, C, tensor_id);
            u_rb = rb;
        }
        return make_float2(sx, u_mine);
    }
    const int64_t n = (int64_t)cb * kTile + (threadIdx.x - kTile);
    return make_float2((A.s_w && n < C.N) ? __ldg(A.s_w + n) : 1.0f, 0.0f);
}

// FOLD: at least one of s_x, s_w is given (a missing one multiplies by 1).
template <int MODE, int FMT, bool FOLD>
__global__ void __launch_bounds__(256, 2)
    quantize_tma_kernel(const __grid_constant__ CUtensorMap tmG, TileQuantArgs A, QuantCommon C, QuantOut O,
                        int64_t ntiles) {
    constexpr int RPT = 8, RS = 16;   // rows r0 + 16 j of the tile, 8 columns from 8 c
    constexpr bool ERR = row_mode(MODE);   // error partials
    extern __shared__ __align__(128) uint8_t qsmem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(qsmem + kQStages * kQTileBytes);
    __shared__ __align__(16) float2 xu_s[3][kTile];   // (s_x, u) per tile row; tile k in slot k % 3
    __shared__ __align__(16) float sw_s[3][kTile];    // s_w per tile column
    __shared__ uint32_t red[2][8];                    // the warps' absmax, tile k in [k & 1]
    __shared__ __align__(16) float col_smem[2][8 * kTile];   // per-warp column sums, tile k in [k & 1]
    const int tid = threadIdx.x, c = tid & 15, r0 = tid >> 4, lane = tid & 31, warp = tid >> 5;
    // tile indices fit 32 bits (checked on the host) and advance incrementally
    const int ntc = (int)C.ntc;
    const int beg = (int)((int64_t)blockIdx.x * ntiles / gridDim.x);
    const int count = (int)(((int64_t)blockIdx.x + 1) * ntiles / gridDim.x) - beg;
    const uint32_t bar0 = (uint32_t)__cvta_generic_to_shared(bars);
    const int64_t row_step = (int64_t)RS * C.N;   // elements between my consecutive rows
    int irb = beg / ntc, icb = beg - (beg / ntc) * ntc;   // next tile to copy (thread 0)
    auto issue = [&](int k) {
        const int s = k % kQStages;
        q_issue_tile((uint32_t)__cvta_generic_to_shared(qsmem + s * kQTileBytes), &tmG, icb * kTile, irb * kTile,
                     bar0 + 8 * s);
        if (++icb == ntc) { icb = 0; ++irb; }
    };
    int rb = beg / ntc, cb = beg - (beg / ntc) * ntc;      // current tile
    int srb = rb, scb = cb;                                // next tile whose side data is fetched
    float u_mine = 0.0f;
    int u_rb = -1;
    auto put_side = [&](int slot, float2 sd) {
        if (tid < kTile) xu_s[slot][tid] = sd;
        else sw_s[slot][tid - kTile] = sd.x;
    };
    for (int i = 0; i < 2 && i < count; ++i) {   // tiles 0 and 1
        put_side(i, q_side<MODE>(A, C, O.tensor_id, srb, scb, u_mine, u_rb));
        if (++scb == ntc) { scb = 0; ++srb; }
    }
    if (tid == 0) {
        for (int i = 0; i < kQStages; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar0 + 8 * i) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmG) : "memory");
    }
    __syncthreads();
    int issued = 0;   // thread 0's count
    if (tid == 0)
        for (; issued < kQStages && issued < count; ++issued) issue(issued);
    int k = 0, s = 0;
    uint32_t phase = 0;
    int prb = 0, pcb = 0;   // the previous tile (its column sums are added one tile later)
    bool done = true;       // false: the CTA left early (a wait ran out)
    for (; k < count; ++k) {
        const int sl = k % 3;
        const int64_t t0 = (int64_t)rb * kTile, n0 = (int64_t)cb * kTile;
        const int nc0 = (int)n0 + 8 * c;
        const int64_t rl = C.T - t0 - r0;
        const int rows_left = rl < kTile ? (int)rl : kTile;   // my row j is valid iff RS j < rows_left
        // side data two tiles ahead: loads (and thresholds) in flight during this tile
        const bool more = k + 2 < count;
        float2 side = make_float2(0.0f, 0.0f);
        if (more) {
            side = q_side<MODE>(A, C, O.tensor_id, srb, scb, u_mine, u_rb);
            if (++scb == ntc) { scb = 0; ++srb; }
        }
        // every thread waits for the tile itself; a wait that ran out is settled at the barrier
        const bool ok = q_wait(bar0 + 8 * s, phase);
        // pass 1: fold g = (s_x * G) * s_w and absmax.  Unscaled input keeps the raw bf16
        // pairs (half the registers) and takes the absmax two at a time in bf16: the
        // magnitude max of a pair of bf16 values is exact, and bf16 -> fp32 is exact.
        float g[FOLD ? RPT : 1][8];
        uint32_t rw[FOLD ? 1 : RPT][4];
        float amax = 0.0f;   // NaN-propagating
        if (!FOLD) {
            const uint16_t* tb = reinterpret_cast<const uint16_t*>(qsmem + s * kQTileBytes);
            uint32_t m2 = 0u;   // |max| per bf16 half (the sign bits are not used)
#pragma unroll
            for (int j = 0; j < RPT; ++j) {
                const uint4 raw = *reinterpret_cast<const uint4*>(tb + (r0 + RS * j) * kTile + 8 * c);
                rw[FOLD ? 0 : j][0] = raw.x; rw[FOLD ? 0 : j][1] = raw.y;
                rw[FOLD ? 0 : j][2] = raw.z; rw[FOLD ? 0 : j][3] = raw.w;
                m2 = bf16x2_absmax_nan(m2, bf16x2_absmax_nan(raw.x, raw.y));
                m2 = bf16x2_absmax_nan(m2, bf16x2_absmax_nan(raw.z, raw.w));
            }
            amax = max3_abs_nan(0.0f, bf16_lo(m2), bf16_hi(m2));
        } else {
            float sw[8];
            if (FOLD) {
                const float4 w0 = *reinterpret_cast<const float4*>(&sw_s[sl][8 * c]);
                const float4 w1 = *reinterpret_cast<const float4*>(&sw_s[sl][8 * c + 4]);
                sw[0] = w0.x; sw[1] = w0.y; sw[2] = w0.z; sw[3] = w0.w;
                sw[4] = w1.x; sw[5] = w1.y; sw[6] = w1.z; sw[7] = w1.w;
            }
            const uint16_t* tb = reinterpret_cast<const uint16_t*>(qsmem + s * kQTileBytes);
#pragma unroll
            for (int j = 0; j < RPT; ++j) {
                const int rr = r0 + RS * j;
                const uint4 raw = *reinterpret_cast<const uint4*>(tb + rr * kTile + 8 * c);
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
                float sx = 1.0f;
                if (FOLD) sx = xu_s[sl][rr].x;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float2 v = make_float2(bf16_lo(w[q]), bf16_hi(w[q]));
                    if (FOLD) {
                        v = f2_mul(v, make_float2(sx, sx));
                        v = f2_mul(v, make_float2(sw[2 * q], sw[2 * q + 1]));
                    }
                    g[FOLD ? j : 0][2 * q] = v.x;
                    g[FOLD ? j : 0][2 * q + 1] = v.y;
                    amax = max3_abs_nan(amax, v.x, v.y);
                }
            }
        }
        // block absmax (non-negative floats and NaN order like their bit patterns)
        {
            const uint32_t wm = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(amax));
            if (lane == 0) red[k & 1][warp] = wm;
        }
        // the one barrier of the tile: every thread is done with this stage (refilled at once),
        // the maxima and the previous tile's column sums are visible, and the CTA leaves
        // together if any wait ran out
        if (!__syncthreads_and(ok)) {
            if (tid == 0) set_status(C.d_status, S3R_ERR_TIMEOUT);
            done = false;
            break;
        }
        if (tid == 0 && issued < count) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(issued);
            ++issued;
        }
        if (ERR && O.col && k > 0 && tid < kTile) {   // the previous tile's column sums, in warp order
            const float* cs = col_smem[(k - 1) & 1];
            float sum = 0.0f;
#pragma unroll
            for (int w = 0; w < 8; ++w) sum += cs[w * kTile + tid];
            if ((int64_t)pcb * kTile + tid < C.N) O.col[(int64_t)prb * C.N + (int64_t)pcb * kTile + tid] = -sum;
        }
        uint32_t amax_bits = __reduce_max_sync(0xFFFFFFFFu, red[k & 1][lane & 7]);
        if (C.tensor_amax) amax_bits = __ldg(C.tensor_amax);   // one step for the whole tensor
        const bool nonfinite = amax_bits >= 0x7F800000u;   // uniform across the CTA
        float d, inv;
        tile_scales(amax_bits, d, inv);
        if (tid == 0) {
            O.scale[(int64_t)rb * ntc + cb] = d;
            if (nonfinite) set_status(C.d_status, S3R_ERR_NONFINITE);
        }
        // pass 2: codes, stores and error sums (of -e, negated when stored)
        float2 colsum[4];
        float rsum[RPT];
        void* q0 = FMT == 0 ? (void*)(static_cast<int8_t*>(O.Q) + (t0 + r0) * C.N + nc0)
                            : (void*)(static_cast<__half*>(O.Q) + (t0 + r0) * C.N + nc0);
        auto gpair = [&](int j, int q) -> float2 {
            if (FOLD) return make_float2(g[FOLD ? j : 0][2 * q], g[FOLD ? j : 0][2 * q + 1]);
            const uint32_t w = rw[FOLD ? 0 : j][q];
            return make_float2(bf16_lo(w), bf16_hi(w));
        };
        round_rows<MODE, FMT, RPT, RS, ERR>(gpair, d, inv, nonfinite, &xu_s[sl][r0].y, 2 * RS, q0, row_step,
                                            rows_left, t0 + r0, nc0, C.N, C.seed_lo, O.tensor_id, rsum, colsum);
        if (ERR && O.tok) {
            const float r = scatter_rows16<RPT>(rsum, c);   // row r0 + 16 (c >> 1)
            if ((c & 1) == 0 && RS * (c >> 1) < rows_left) O.tok[(t0 + r0 + RS * (c >> 1)) * ntc + cb] = -r;
        }
        if (ERR && O.col) {
            float cs[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                cs[2 * q] = colsum[q].x + __shfl_xor_sync(0xFFFFFFFFu, colsum[q].x, 16);
                cs[2 * q + 1] = colsum[q].y + __shfl_xor_sync(0xFFFFFFFFu, colsum[q].y, 16);
            }
            if (lane < 16) {
                float* dst = &col_smem[k & 1][warp * kTile + 8 * c];
                *reinterpret_cast<float4*>(dst) = make_float4(cs[0], cs[1], cs[2], cs[3]);
                *reinterpret_cast<float4*>(dst + 4) = make_float4(cs[4], cs[5], cs[6], cs[7]);
            }
        }
        // slot (k + 2) % 3 held the previous tile's side data, which every thread finished
        // reading before this tile's barrier
        if (more) put_side((k + 2) % 3, side);
        prb = rb;
        pcb = cb;
        if (++cb == ntc) { cb = 0; ++rb; }
        if (++s == kQStages) { s = 0; phase ^= 1u; }
    }
    if (done && count > 0 && ERR && O.col) {   // the last tile's column sums
        __syncthreads();
        if (tid < kTile) {
            const float* cs = col_smem[(count - 1) & 1];
            float sum = 0.0f;
#pragma unroll
            for (int w = 0; w < 8; ++w) sum += cs[w * kTile + tid];
            if ((int64_t)pcb * kTile + tid < C.N) O.col[(int64_t)prb * C.N + (int64_t)pcb * kTile + tid] = -sum;
        }
    }
    // an early exit may leave copies in flight: wait for them before leaving
    if (tid == 0)
        for (int q = k; q < issued; ++q) q_wait(bar0 + 8 * (q % kQStages), (uint32_t)((q / kQStages) & 1));
}

// ---------------------------------------------------------------------------
// SwiGLU glue fused into the two quantizations (dh1 -> Q1, dh3 -> Q3).
// ---------------------------------------------------------------------------
struct SwigluArgs {
    const float* dA;
    int64_t ldd;
    const uint16_t* h1;
    const uint16_t* h3;
    int64_t ldh;
    const float* s_x;
    const float* s_w1;
    const float* s_w3;
    bool vec_load;
};

// Block-wide max of two values (non-negative float bit patterns, NaN largest).
template <int WARPS>
__device__ __forceinline__ void block_max2_u32(uint32_t& a, uint32_t& b, uint32_t* smem /* [2][WARPS] */) {
    a = __reduce_max_sync(0xFFFFFFFFu, a);
    b = __reduce_max_sync(0xFFFFFFFFu, b);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        smem[warp] = a;
        smem[WARPS + warp] = b;
    }
    __syncthreads();
    uint32_t ma = 0, mb = 0;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
        ma = max(ma, smem[w]);
        mb = max(mb, smem[WARPS + w]);
    }
    __syncthreads();
    a = ma;
    b = mb;
}

// One 128x128 tile of the SwiGLU glue and its two quantizations; 512
// threads, each 4 rows x 8 columns.  SMEM: the tile's dA (fp32) and h1, h3
// (bf16) rows come from shared memory (pitch 128 elements) instead of global
// memory; `freed` runs once every thread is done reading them.
template <int MODE, bool SMEM, typename Freed>
__device__ __forceinline__ void swiglu_tile(const SwigluArgs& A, const QuantCommon& C, const QuantOut& O1,
                                            const QuantOut& O3, int64_t t0, int64_t n0, const float* sd,
                                            const uint16_t* s1, const uint16_t* s3, uint32_t* red, float* col_smem,
                                            Freed freed) {
    constexpr int RPT = 4;
    using Geo = TileGeom<RPT>;
    const int c = threadIdx.x & 15, r0 = threadIdx.x >> 4;
    const int64_t nc0 = n0 + 8 * c;

    float g1[RPT][8], g3[RPT][8];
    float sw1[8], sw3[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const bool ok = nc0 + i < C.N;
        sw1[i] = (A.s_w1 && ok) ? __ldg(A.s_w1 + nc0 + i) : 1.0f;
        sw3[i] = (A.s_w3 && ok) ? __ldg(A.s_w3 + nc0 + i) : 1.0f;
    }
    float am1 = 0.0f, am3 = 0.0f;   // NaN-propagating absmax of each tile
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
        const int rr = r0 + j * Geo::kRowStride;
        const int64_t t = t0 + rr;
        float da[8], x1[8], x3[8];
        if (SMEM) {
            // the copy zero-fills outside the tensor
            const float4 d0 = *reinterpret_cast<const float4*>(sd + rr * kTile + 8 * c);
            const float4 d1 = *reinterpret_cast<const float4*>(sd + rr * kTile + 8 * c + 4);
            const uint4 a1 = *reinterpret_cast<const uint4*>(s1 + rr * kTile + 8 * c);
            const uint4 a3 = *reinterpret_cast<const uint4*>(s3 + rr * kTile + 8 * c);
            da[0] = d0.x; da[1] = d0.y; da[2] = d0.z; da[3] = d0.w;
            da[4] = d1.x; da[5] = d1.y; da[6] = d1.z; da[7] = d1.w;
            const uint32_t w1[4] = {a1.x, a1.y, a1.z, a1.w}, w3[4] = {a3.x, a3.y, a3.z, a3.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                x1[i] = (i & 1) ? bf16_hi(w1[i >> 1]) : bf16_lo(w1[i >> 1]);
                x3[i] = (i & 1) ? bf16_hi(w3[i >> 1]) : bf16_lo(w3[i >> 1]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) da[i] = x1[i] = x3[i] = 0.0f;
            if (t < C.T) {
                const float* pd = A.dA + t * A.ldd + nc0;
                const uint16_t* p1 = A.h1 + t * A.ldh + nc0;
                const uint16_t* p3 = A.h3 + t * A.ldh + nc0;
                if (A.vec_load && nc0 + 8 <= C.N) {
                    const float4 d0 = __ldg(reinterpret_cast<const float4*>(pd));
                    const float4 d1 = __ldg(reinterpret_cast<const float4*>(pd) + 1);
                    const uint4 a1 = __ldg(reinterpret_cast<const uint4*>(p1));
                    const uint4 a3 = __ldg(reinterpret_cast<const uint4*>(p3));
                    da[0] = d0.x; da[1] = d0.y; da[2] = d0.z; da[3] = d0.w;
                    da[4] = d1.x; da[5] = d1.y; da[6] = d1.z; da[7] = d1.w;
                    const uint32_t w1[4] = {a1.x, a1.y, a1.z, a1.w}, w3[4] = {a3.x, a3.y, a3.z, a3.w};
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        x1[i] = (i & 1) ? bf16_hi(w1[i >> 1]) : bf16_lo(w1[i >> 1]);
                        x3[i] = (i & 1) ? bf16_hi(w3[i >> 1]) : bf16_lo(w3[i >> 1]);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (nc0 + i < C.N) {
                            da[i] = pd[i];
                            x1[i] = bf16_at(p1 + i);
                            x3[i] = bf16_at(p3 + i);
                        }
                }
            }
        }
        const float sx = (A.s_x && t < C.T) ? __ldg(A.s_x + t) : 1.0f;
        // negated folds: (-s_x) * dh * s_w == -((s_x * dh) * s_w) exactly
        const float nsx = A.s_x ? -sx : -1.0f;
        const float2 nsx2 = make_float2(nsx, nsx);
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            // glue, in the documented order, two lanes per packed instruction
            // (no contraction: built with -fmad=false)
            const float2 x = make_float2(x1[i], x1[i + 1]);
            const float2 d2 = make_float2(da[i], da[i + 1]);
            float2 silu, dsilu;
            swiglu_terms2(x, silu, dsilu);
            const float2 dh1 = f2_mul(f2_mul(d2, make_float2(x3[i], x3[i + 1])), dsilu);
            const float2 dh3 = f2_mul(d2, silu);
            float2 v1 = f2_mul(nsx2, dh1), v3 = f2_mul(nsx2, dh3);
            if (A.s_w1) v1 = f2_mul(v1, make_float2(sw1[i], sw1[i + 1]));
            if (A.s_w3) v3 = f2_mul(v3, make_float2(sw3[i], sw3[i + 1]));
            g1[j][i] = v1.x;
            g1[j][i + 1] = v1.y;
            g3[j][i] = v3.x;
            g3[j][i + 1] = v3.y;
            am1 = max3_abs_nan(am1, v1.x, v1.y);
            am3 = max3_abs_nan(am3, v3.x, v3.y);
        }
    }
    // non-negative floats and NaN order like their bit patterns; after the
    // reduction's barriers no thread reads the staged tile any more
    uint32_t amax1 = __float_as_uint(am1), amax3 = __float_as_uint(am3);
    block_max2_u32<Geo::kWarps>(amax1, amax3, red);
    freed();
    round_and_store<MODE, RPT>(g1, amax1, t0, n0, r0, c, C, O1, col_smem);
    round_and_store<MODE, RPT>(g3, amax3, t0, n0, r0, c, C, O3, col_smem);
}

template <int MODE>
__global__ void __launch_bounds__(512) swiglu_quantize_kernel(SwigluArgs A, QuantCommon C, QuantOut O1, QuantOut O3) {
    __shared__ uint32_t red[2 * 16];
    __shared__ float col_smem[16 * 128];
    swiglu_tile<MODE, false>(A, C, O1, O3, (int64_t)blockIdx.y * kTile, (int64_t)blockIdx.x * kTile, nullptr, nullptr,
                             nullptr, red, col_smem, [] {});
}

// Persistent variant: one CTA per SM walks tiles tile = blockIdx.x + i * gridDim.x.
// TMA copies the next tile's dA (fp32) and h1, h3 (bf16) into shared memory
// (128 KB) while the current tile is quantized from registers, so the HBM
// stream is not exposed between tiles.

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Persistent SwiGLU quantizer: CTA b owns a contiguous range of 128 x 128
// tiles in row-major order (consecutive tiles share a row block and its two
// threshold sets).  Each tile arrives as four 32-row quarters (dA fp32, h1 and
// h3 bf16: 32 KiB) through a six-quarter TMA ring, so one and a half tiles are
// in flight while one is rounded; thread (c, r0) owns row r0 + 32 j of quarter
// j and columns 8c .. 8c + 7.  The side data of a tile (row scale and the two
// row thresholds; the two column scales) is fetched one tile ahead.
constexpr int kSwQuarterRows = 32;
constexpr int kSwQuarterBytes = kSwQuarterRows * kTile * (4 + 2 + 2);   // 32 KiB
constexpr int kSwStages = 6;
constexpr int kSwigluTmaSmem = kSwStages * kSwQuarterBytes + 8 * kSwStages + 128;

template <int MODE>
__device__ __forceinline__ void sw_side(const SwigluArgs& A, const QuantCommon& C, const QuantOut& O1,
                                        const QuantOut& O3, int rb, int cb, float4& xs, float2& ws, float& u1,
                                        float& u3, int& u_rb) {
    if (threadIdx.x < kTile) {
        const int64_t t = (int64_t)rb * kTile + threadIdx.x;
        const float sx = (A.s_x && t < C.T) ? __ldg(A.s_x + t) : 1.0f;
        if (row_mode(MODE) && rb != u_rb) {
            u1 = row_threshold<MODE>((uint64_t)t, C, O1.tensor_id);
            u3 = row_threshold<MODE>((uint64_t)t, C, O3.tensor_id);
            u_rb = rb;
        }
        xs = make_float4(sx, u1, u3, 0.0f);
    } else if (threadIdx.x < 2 * kTile) {
        const int64_t n = (int64_t)cb * kTile + (threadIdx.x - kTile);
        const bool ok = n < C.N;
        ws = make_float2((A.s_w1 && ok) ? __ldg(A.s_w1 + n) : 1.0f, (A.s_w3 && ok) ? __ldg(A.s_w3 + n) : 1.0f);
    }
}

template <int MODE, int FMT>
__global__ void __launch_bounds__(512, 1)
    swiglu_tma_kernel(const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmH1,
                      const __grid_constant__ CUtensorMap tmH3, SwigluArgs A, QuantCommon C, QuantOut O1, QuantOut O3,
                      int64_t ntiles) {
    constexpr int RPT = 4, RS = 32;
    constexpr bool ERR = row_mode(MODE);
    extern __shared__ uint8_t swsm_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(swsm_raw) + 127) & ~(uintptr_t)127);
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring + kSwStages * kSwQuarterBytes);
    __shared__ __align__(16) float4 xs_s[2][kTile];   // (s_x, u1, u3, 0) per tile row
    __shared__ __align__(16) float2 ws_s[2][kTile];   // (s_w1, s_w3) per tile column
    __shared__ uint32_t red[2][16];
    __shared__ __align__(16) float col_smem[2][16 * kTile];
    const int tid = threadIdx.x, c = tid & 15, r0 = tid >> 4, lane = tid & 31, warp = tid >> 5;
    const int ntc = (int)C.ntc;
    const int beg = (int)((int64_t)blockIdx.x * ntiles / gridDim.x);
    const int count = (int)(((int64_t)blockIdx.x + 1) * ntiles / gridDim.x) - beg;
    const int nq = 4 * count;   // quarters this CTA streams
    const uint32_t bar0 = (uint32_t)__cvta_generic_to_shared(bars);
    const int64_t row_step = (int64_t)RS * C.N;
    int irb = beg / ntc, icb = beg - (beg / ntc) * ntc, iq = 0;   // next quarter to copy (thread 0)
    auto issue = [&](int q) {
        const int st = q % kSwStages;
        const uint32_t bar = bar0 + 8 * st;
        uint8_t* dst = ring + st * kSwQuarterBytes;
        const int32_t x = icb * kTile, y = irb * kTile + iq * kSwQuarterRows;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(kSwQuarterBytes)
                     : "memory");
        tma_2d((uint32_t)__cvta_generic_to_shared(dst), &tmD, x, y, bar);
        tma_2d((uint32_t)__cvta_generic_to_shared(dst + kSwQuarterRows * kTile * 4), &tmH1, x, y, bar);
        tma_2d((uint32_t)__cvta_generic_to_shared(dst + kSwQuarterRows * kTile * 6), &tmH3, x, y, bar);
        if (++iq == 4) {
            iq = 0;
            if (++icb == ntc) { icb = 0; ++irb; }
        }
    };
    int rb = beg / ntc, cb = beg - (beg / ntc) * ntc;
    int nrb = rb, ncb = cb;
    if (++ncb == ntc) { ncb = 0; ++nrb; }
    float u1 = 0.0f, u3 = 0.0f;
    int u_rb = -1;
    {
        float4 xs = make_float4(0.f, 0.f, 0.f, 0.f);
        float2 ws = make_float2(0.f, 0.f);
        if (count > 0) sw_side<MODE>(A, C, O1, O3, rb, cb, xs, ws, u1, u3, u_rb);
        if (tid < kTile) xs_s[0][tid] = xs;
        else if (tid < 2 * kTile) ws_s[0][tid - kTile] = ws;
    }
    if (tid == 0) {
        for (int i = 0; i < kSwStages; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar0 + 8 * i) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmD) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmH1) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmH3) : "memory");
    }
    __syncthreads();
    int issued = 0;   // quarters copied (thread 0's count)
    if (tid == 0)
        for (; issued < kSwStages && issued < nq; ++issued) issue(issued);
    int k = 0;
    for (; k < count; ++k) {
        const int sl = k & 1;
        const int64_t t0 = (int64_t)rb * kTile, n0 = (int64_t)cb * kTile;
        const int nc0 = (int)n0 + 8 * c;
        const int64_t rl = C.T - t0 - r0;
        const int rows_left = rl < kTile ? (int)rl : kTile;
        float4 nxs = make_float4(0.f, 0.f, 0.f, 0.f);
        float2 nws = make_float2(0.f, 0.f);
        if (k + 1 < count) sw_side<MODE>(A, C, O1, O3, nrb, ncb, nxs, nws, u1, u3, u_rb);
        // pass 1: glue and folds, quarter by quarter.  Each thread waits for its
        // quarters itself; a wait that ran out is settled at the next barrier.
        float g1[RPT][8], g3[RPT][8];
        float am1 = 0.0f, am3 = 0.0f;   // NaN-propagating absmax of each tile
        bool ok = true;
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            const int q = 4 * k + j, st = q % kSwStages;
            ok = ok && q_wait(bar0 + 8 * st, (uint32_t)((q / kSwStages) & 1));
            const uint8_t* base = ring + st * kSwQuarterBytes;
            const float* sd = reinterpret_cast<const float*>(base) + r0 * kTile + 8 * c;
            const uint16_t* s1 = reinterpret_cast<const uint16_t*>(base + kSwQuarterRows * kTile * 4) + r0 * kTile + 8 * c;
            const uint16_t* s3 = reinterpret_cast<const uint16_t*>(base + kSwQuarterRows * kTile * 6) + r0 * kTile + 8 * c;
            const float4 d0 = *reinterpret_cast<const float4*>(sd);
            const float4 d1 = *reinterpret_cast<const float4*>(sd + 4);
            const uint4 a1 = *reinterpret_cast<const uint4*>(s1);
            const uint4 a3 = *reinterpret_cast<const uint4*>(s3);
            const float da[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
            const uint32_t h1w[4] = {a1.x, a1.y, a1.z, a1.w}, h3w[4] = {a3.x, a3.y, a3.z, a3.w};
            const float sx = xs_s[sl][r0 + RS * j].x;
            const float2 sx2 = make_float2(sx, sx);
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
                // glue, in the documented order, two lanes per packed instruction
                // (no contraction: built with -fmad=false)
                const float2 x = make_float2(bf16_lo(h1w[i >> 1]), bf16_hi(h1w[i >> 1]));
                const float2 x3 = make_float2(bf16_lo(h3w[i >> 1]), bf16_hi(h3w[i >> 1]));
                const float2 d2 = make_float2(da[i], da[i + 1]);
                float2 silu, dsilu;
                swiglu_terms2(x, silu, dsilu);
                const float2 dh1 = f2_mul(f2_mul(d2, x3), dsilu);
                const float2 dh3 = f2_mul(d2, silu);
                // folds (s_x * dh) * s_w; a missing scale is 1
                const float4 wp = *reinterpret_cast<const float4*>(&ws_s[sl][8 * c + i]);   // (w1, w3) of i, i + 1
                const float2 v1 = f2_mul(f2_mul(sx2, dh1), make_float2(wp.x, wp.z));
                const float2 v3 = f2_mul(f2_mul(sx2, dh3), make_float2(wp.y, wp.w));
                g1[j][i] = v1.x;
                g1[j][i + 1] = v1.y;
                g3[j][i] = v3.x;
                g3[j][i + 1] = v3.y;
                am1 = max3_abs_nan(am1, v1.x, v1.y);
                am3 = max3_abs_nan(am3, v3.x, v3.y);
            }
        }
        {
            const uint32_t m1 = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(am1));
            const uint32_t m3 = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(am3));
            if (lane == 0) {
                red[0][warp] = m1;
                red[1][warp] = m3;
            }
        }
        // every thread is done with this tile's quarters; the CTA leaves together if a wait ran out
        if (!__syncthreads_and(ok)) {
            if (tid == 0) set_status(C.d_status, S3R_ERR_TIMEOUT);
            break;
        }
        if (tid == 0 && issued < nq) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            for (int i = 0; i < 4 && issued < nq; ++i, ++issued) issue(issued);
        }
        const uint32_t amax1 = __reduce_max_sync(0xFFFFFFFFu, red[0][lane & 15]);
        const uint32_t amax3 = __reduce_max_sync(0xFFFFFFFFu, red[1][lane & 15]);
        // lanes 0 and 1 derive the two tiles' scales side by side
        float dd, ii;
        tile_scales((lane & 1) ? amax3 : amax1, dd, ii);
        const float d1s = __shfl_sync(0xFFFFFFFFu, dd, 0), inv1 = __shfl_sync(0xFFFFFFFFu, ii, 0);
        const float d3s = __shfl_sync(0xFFFFFFFFu, dd, 1), inv3 = __shfl_sync(0xFFFFFFFFu, ii, 1);
        const bool nf1 = amax1 >= 0x7F800000u, nf3 = amax3 >= 0x7F800000u;   // uniform across the CTA
        if (tid == 0) {
            O1.scale[(int64_t)rb * ntc + cb] = d1s;
            O3.scale[(int64_t)rb * ntc + cb] = d3s;
            if (nf1 || nf3) set_status(C.d_status, S3R_ERR_NONFINITE);
        }
        // pass 2: codes, stores and error sums (of -e, negated when stored)
        const int64_t off = (t0 + r0) * C.N + nc0;
#pragma unroll
        for (int o = 0; o < 2; ++o) {
            const QuantOut& O = o ? O3 : O1;
            float2 colsum[4];
            float rsum[RPT];
            void* q0 = FMT == 0 ? (void*)(static_cast<int8_t*>(O.Q) + off) : (void*)(static_cast<__half*>(O.Q) + off);
            auto gpair = [&](int j, int q) -> float2 {
                return o ? make_float2(g3[j][2 * q], g3[j][2 * q + 1]) : make_float2(g1[j][2 * q], g1[j][2 * q + 1]);
            };
            round_rows<MODE, FMT, RPT, RS, ERR>(gpair, o ? d3s : d1s, o ? inv3 : inv1, o ? nf3 : nf1,
                                                o ? &xs_s[sl][r0].z : &xs_s[sl][r0].y, 4 * RS, q0, row_step,
                                                rows_left, t0 + r0, nc0, C.N, C.seed_lo, O.tensor_id, rsum, colsum);
            if (ERR && O.tok) {
                const float r = scatter_rows16<RPT>(rsum, c);   // row r0 + 32 (c >> 2)
                if ((c & 3) == 0 && RS * (c >> 2) < rows_left) O.tok[(t0 + r0 + RS * (c >> 2)) * ntc + cb] = -r;
            }
            if (ERR && O.col) {
                float cs[8];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    cs[2 * q] = colsum[q].x + __shfl_xor_sync(0xFFFFFFFFu, colsum[q].x, 16);
                    cs[2 * q + 1] = colsum[q].y + __shfl_xor_sync(0xFFFFFFFFu, colsum[q].y, 16);
                }
                if (lane < 16) {
                    float* dst = &col_smem[o][warp * kTile + 8 * c];
                    *reinterpret_cast<float4*>(dst) = make_float4(cs[0], cs[1], cs[2], cs[3]);
                    *reinterpret_cast<float4*>(dst + 4) = make_float4(cs[4], cs[5], cs[6], cs[7]);
                }
            }
        }
        if (k + 1 < count) {
            if (tid < kTile) xs_s[sl ^ 1][tid] = nxs;
            else if (tid < 2 * kTile) ws_s[sl ^ 1][tid - kTile] = nws;
        }
        __syncthreads();
        if (ERR && tid < 2 * kTile) {
            const int o = tid >> 7, n = tid & (kTile - 1);
            const QuantOut& O = o ? O3 : O1;
            if (O.col) {
                float sum = 0.0f;
#pragma unroll
                for (int w = 0; w < 16; ++w) sum += col_smem[o][w * kTile + n];
                if (n0 + n < C.N) O.col[(int64_t)rb * C.N + n0 + n] = -sum;
            }
        }
        rb = nrb;
        cb = ncb;
        if (++ncb == ntc) { ncb = 0; ++nrb; }
    }
    // an early exit may leave copies in flight: wait for them before leaving
    if (tid == 0)
        for (int q = 4 * k; q < issued; ++q) q_wait(bar0 + 8 * (q % kSwStages), (uint32_t)((q / kSwStages) & 1));
}

// ---------------------------------------------------------------------------
// Forward operands: RTNE with one scale per row or per column (scale 1 for an
// all-zero row/column).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void store_code(void* Q, int fmt, int64_t idx, float q) {
    if (fmt == S3R_CODES_S8) static_cast<int8_t*>(Q)[idx] = (int8_t)(int)q;
    else static_cast<__half*>(Q)[idx] = __int2half_rn((int)q);
}

__global__ void __launch_bounds__(256) rtne_rows_kernel(const uint16_t* A, int64_t R, int64_t C, int64_t lda,
                                                        void* Q, int fmt, float* scale, int* d_status) {
    const int64_t r = (int64_t)blockIdx.x;
    __shared__ uint32_t red[8];
    uint32_t m = 0u;
    for (int64_t c = threadIdx.x; c < C; c += blockDim.x)
        m = max(m, __float_as_uint(bf16_at(A + r * lda + c)) & 0x7FFFFFFFu);
    m = block_max_u32<8>(m, red);
    if (m >= 0x7F800000u) {
        if (threadIdx.x == 0) { set_status(d_status, S3R_ERR_NONFINITE); scale[r] = __uint_as_float(0x7FC00000u); }
        for (int64_t c = threadIdx.x; c < C; c += blockDim.x) store_code(Q, fmt, r * C + c, 0.0f);
        return;
    }
    const float amax = __uint_as_float(m);
    const float s = m ? amax / 127.0f : 1.0f;
    const float inv = m ? __fdiv_rz(127.0f, amax) : 1.0f;   // |a * inv| <= 127
    if (threadIdx.x == 0) scale[r] = s;
    for (int64_t c = threadIdx.x; c < C; c += blockDim.x) {
        const float q = fminf(fmaxf(rintf(bf16_at(A + r * lda + c) * inv), -127.0f), 127.0f);
        store_code(Q, fmt, r * C + c, q);
    }
}

__global__ void __launch_bounds__(256) rtne_cols_kernel(const uint16_t* A, int64_t R, int64_t C, int64_t lda,
                                                        void* Q, int fmt, float* scale, int* d_status) {
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= C) return;
    uint32_t m = 0u;
    for (int64_t r = 0; r < R; ++r) m = max(m, __float_as_uint(bf16_at(A + r * lda + c)) & 0x7FFFFFFFu);
    if (m >= 0x7F800000u) {
        set_status(d_status, S3R_ERR_NONFINITE);
        scale[c] = __uint_as_float(0x7FC00000u);
        for (int64_t r = 0; r < R; ++r) store_code(Q, fmt, r * C + c, 0.0f);
        return;
    }
    const float amax = __uint_as_float(m);
    const float s = m ? amax / 127.0f : 1.0f;
    const float inv = m ? __fdiv_rz(127.0f, amax) : 1.0f;   // |a * inv| <= 127
    scale[c] = s;
    for (int64_t r = 0; r < R; ++r) {
        const float q = fminf(fmaxf(rintf(bf16_at(A + r * lda + c) * inv), -127.0f), 127.0f);
        store_code(Q, fmt, r * C + c, q);
    }
}

// Vectorized forms for 16-byte aligned rows (C and lda multiples of 8): the
// same arithmetic element by element, on 8 bf16 values per 16-byte access.

// max of |x| over 8 bf16 as a float bit pattern (NaN/Inf compare largest)
__device__ __forceinline__ uint32_t absmax8_bits(const uint4& v) {
    uint32_t m = __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu), __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
    return max(m & 0xFFFFu, m >> 16) << 16;
}

// 8 codes of one 16-byte group: q = clamp(rint(a * inv[i]), -127, 127)
template <int FMT>
__device__ __forceinline__ void store_codes8(void* Q, int64_t idx, const uint4& v, const float (&inv)[8],
                                             bool zero) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float a = __uint_as_float(i & 1 ? (w[i >> 1] & 0xFFFF0000u) : (w[i >> 1] << 16));
        q[i] = zero ? 0.0f : fminf(fmaxf(rintf(a * inv[i]), -127.0f), 127.0f);
    }
    if (FMT == S3R_CODES_F16) {
        uint32_t h[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 p = __floats2half2_rn(q[2 * i], q[2 * i + 1]);
            h[i] = *reinterpret_cast<const uint32_t*>(&p);
        }
        *reinterpret_cast<uint4*>(static_cast<__half*>(Q) + idx) = make_uint4(h[0], h[1], h[2], h[3]);
    } else {
        uint32_t b[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 8; ++i) b[i >> 2] |= ((uint32_t)(int)q[i] & 0xFFu) << (8 * (i & 3));
        *reinterpret_cast<uint2*>(static_cast<int8_t*>(Q) + idx) = make_uint2(b[0], b[1]);
    }
}

// Block-wide max over a block of `blockDim.x / 32` warps (at most 8).
__device__ __forceinline__ uint32_t block_max_dyn(uint32_t v, uint32_t* smem) {
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) smem[warp] = v;
    __syncthreads();
    uint32_t m = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = max(m, smem[w]);
    return m;
}

// Rows of 16-byte groups: one row per block of 32 * ceil(groups / 128) threads
// (at most 256), so that each thread holds up to kRowRegs groups between the
// max and the rounding; longer rows are read again (or recomputed).
constexpr int kRowRegs = 4;

static inline unsigned row_block_threads(int64_t groups) {
    const int64_t w = (groups + 32 * kRowRegs - 1) / (32 * kRowRegs);
    return (unsigned)(32 * (w < 1 ? 1 : (w > 8 ? 8 : w)));
}

// The row's step and 1/step from its max bits; a non-finite row gets a NaN
// step, zero codes and the status flag.
__device__ __forceinline__ float row_scale_finish(uint32_t m, int64_t r, float* scale, int* d_status, bool& bad) {
    bad = m >= 0x7F800000u;
    const float amax = __uint_as_float(m);
    if (threadIdx.x == 0) {
        scale[r] = bad ? __uint_as_float(0x7FC00000u) : (m ? amax / 127.0f : 1.0f);
        if (bad) set_status(d_status, S3R_ERR_NONFINITE);
    }
    return bad ? 0.0f : (m ? __fdiv_rz(127.0f, amax) : 1.0f);   // |a * inv| <= 127
}

template <int FMT>
__global__ void __launch_bounds__(256) rtne_rows_vec_kernel(const uint16_t* A, int64_t C, int64_t lda, void* Q,
                                                            float* scale, int* d_status) {
    __shared__ uint32_t red[8];
    const int64_t r = (int64_t)blockIdx.x;
    const int nt = (int)blockDim.x;
    const uint4* row = reinterpret_cast<const uint4*>(A + r * lda);
    const int64_t nv = C / 8;
    uint4 v[kRowRegs];
    uint32_t m = 0u;
#pragma unroll
    for (int i = 0; i < kRowRegs; ++i) {
        const int64_t j = threadIdx.x + (int64_t)nt * i;
        v[i] = j < nv ? __ldg(row + j) : make_uint4(0u, 0u, 0u, 0u);
        m = max(m, absmax8_bits(v[i]));
    }
    for (int64_t j = threadIdx.x + (int64_t)nt * kRowRegs; j < nv; j += nt) m = max(m, absmax8_bits(__ldg(row + j)));
    bool bad;
    const float iv = row_scale_finish(block_max_dyn(m, red), r, scale, d_status, bad);
    const float inv[8] = {iv, iv, iv, iv, iv, iv, iv, iv};
#pragma unroll
    for (int i = 0; i < kRowRegs; ++i) {
        const int64_t j = threadIdx.x + (int64_t)nt * i;
        if (j < nv) store_codes8<FMT>(Q, r * C + 8 * j, v[i], inv, bad);
    }
    for (int64_t j = threadIdx.x + (int64_t)nt * kRowRegs; j < nv; j += nt)
        store_codes8<FMT>(Q, r * C + 8 * j, __ldg(row + j), inv, bad);
}

// The forward SwiGLU gate fused into the per-row RTNE of its output: from
// bf16 h1 and h3, a = bf16((h1 * sigmoid(h1)) * h3) element by element (fp32,
// that order), then the row's step max|a| / 127 and codes exactly as
// rtne_rows_vec_kernel on a.
__device__ __forceinline__ uint4 swiglu_gate8(const uint4& h1, const uint4& h3) {
    const uint32_t x2[4] = {h1.x, h1.y, h1.z, h1.w}, z2[4] = {h3.x, h3.y, h3.z, h3.w};
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 x = make_float2(__uint_as_float(x2[k] << 16), __uint_as_float(x2[k] & 0xFFFF0000u));
        const float2 z = make_float2(__uint_as_float(z2[k] << 16), __uint_as_float(z2[k] & 0xFFFF0000u));
        const float2 a = f2_mul(f2_mul(x, sigmoid2(x)), z);
        const __nv_bfloat162 p = __floats2bfloat162_rn(a.x, a.y);
        w[k] = *reinterpret_cast<const uint32_t*>(&p);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int FMT>
__global__ void __launch_bounds__(256) swiglu_fwd_rows_kernel(const uint16_t* H1, const uint16_t* H3, int64_t F,
                                                              int64_t ldh, uint16_t* Aout, void* Q, float* scale,
                                                              int* d_status) {
    __shared__ uint32_t red[8];
    const int64_t r = (int64_t)blockIdx.x;
    const int nt = (int)blockDim.x;
    const uint4* h1 = reinterpret_cast<const uint4*>(H1 + r * ldh);
    const uint4* h3 = reinterpret_cast<const uint4*>(H3 + r * ldh);
    const int64_t nv = F / 8;
    uint4 v[kRowRegs];
    uint32_t m = 0u;
#pragma unroll
    for (int i = 0; i < kRowRegs; ++i) {
        const int64_t j = threadIdx.x + (int64_t)nt * i;
        v[i] = j < nv ? swiglu_gate8(__ldg(h1 + j), __ldg(h3 + j)) : make_uint4(0u, 0u, 0u, 0u);
        m = max(m, absmax8_bits(v[i]));
        if (Aout && j < nv) *reinterpret_cast<uint4*>(Aout + r * F + 8 * j) = v[i];
    }
    for (int64_t j = threadIdx.x + (int64_t)nt * kRowRegs; j < nv; j += nt) {
        const uint4 a = swiglu_gate8(__ldg(h1 + j), __ldg(h3 + j));
        m = max(m, absmax8_bits(a));
        if (Aout) *reinterpret_cast<uint4*>(Aout + r * F + 8 * j) = a;
    }
    bool bad;
    const float iv = row_scale_finish(block_max_dyn(m, red), r, scale, d_status, bad);
    const float inv[8] = {iv, iv, iv, iv, iv, iv, iv, iv};
#pragma unroll
    for (int i = 0; i < kRowRegs; ++i) {
        const int64_t j = threadIdx.x + (int64_t)nt * i;
        if (j < nv) store_codes8<FMT>(Q, r * F + 8 * j, v[i], inv, bad);
    }
    for (int64_t j = threadIdx.x + (int64_t)nt * kRowRegs; j < nv; j += nt)
        store_codes8<FMT>(Q, r * F + 8 * j, swiglu_gate8(__ldg(h1 + j), __ldg(h3 + j)), inv, bad);
}

// Per-column scales in three stream-ordered launches: the column maxima
// (atomicMax of the bit patterns into `bits`, zeroed before), the rounding
// with 1/step from those maxima, then bits -> scale.  Blocks take 64 columns
// x 256 rows: thread t reads 8 columns (16 bytes) of rows t/8, t/8 + 32, ...
constexpr int kColStrip = 64, kColChunk = 256;

__global__ void __launch_bounds__(256) rtne_colmax_kernel(const uint16_t* A, int64_t R, int64_t C, int64_t lda,
                                                          uint32_t* bits) {
    __shared__ uint32_t part[32][33];
    const int g = threadIdx.x & 7, rr = threadIdx.x >> 3;
    const int64_t c0 = (int64_t)blockIdx.x * kColStrip + 8 * g;
    const int64_t r0 = (int64_t)blockIdx.y * kColChunk;
    uint32_t m[4] = {0u, 0u, 0u, 0u};
    if (c0 < C) {
#pragma unroll 4
        for (int k = 0; k < kColChunk / 32; ++k) {
            const int64_t r = r0 + rr + 32 * k;
            if (r < R) {
                const uint4 v = __ldg(reinterpret_cast<const uint4*>(A + r * lda + c0));
                m[0] = __vmaxu2(m[0], v.x & 0x7FFF7FFFu);
                m[1] = __vmaxu2(m[1], v.y & 0x7FFF7FFFu);
                m[2] = __vmaxu2(m[2], v.z & 0x7FFF7FFFu);
                m[3] = __vmaxu2(m[3], v.w & 0x7FFF7FFFu);
            }
        }
    }
#pragma unroll
    for (int w = 0; w < 4; ++w) part[rr][4 * g + w] = m[w];
    __syncthreads();
    if (threadIdx.x < 32) {   // one word (two columns) per thread, over the 32 row slots
        uint32_t x = 0u;
        for (int k = 0; k < 32; ++k) x = __vmaxu2(x, part[k][threadIdx.x]);
        const int64_t c = (int64_t)blockIdx.x * kColStrip + 2 * threadIdx.x;
        if (c < C) atomicMax(bits + c, (x & 0xFFFFu) << 16);
        if (c + 1 < C) atomicMax(bits + c + 1, x & 0xFFFF0000u);
    }
}

template <int FMT>
__global__ void __launch_bounds__(256) rtne_cols_vec_kernel(const uint16_t* A, int64_t R, int64_t C, int64_t lda,
                                                            void* Q, const uint32_t* bits, int* d_status) {
    const int g = threadIdx.x & 7, rr = threadIdx.x >> 3;
    const int64_t c0 = (int64_t)blockIdx.x * kColStrip + 8 * g;
    const int64_t r0 = (int64_t)blockIdx.y * kColChunk;
    if (c0 >= C) return;
    float inv[8];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t m = __ldg(bits + c0 + i);
        bad = bad || m >= 0x7F800000u;
        inv[i] = m >= 0x7F800000u ? 0.0f : (m ? __fdiv_rz(127.0f, __uint_as_float(m)) : 1.0f);
    }
    if (bad && blockIdx.y == 0 && rr == 0) set_status(d_status, S3R_ERR_NONFINITE);
#pragma unroll 4
    for (int k = 0; k < kColChunk / 32; ++k) {
        const int64_t r = r0 + rr + 32 * k;
        if (r < R) {
            uint4 v = __ldg(reinterpret_cast<const uint4*>(A + r * lda + c0));
            if (bad) {   // a non-finite column codes to 0: mask its values (inv = 0 would give NaN * 0)
                uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (inv[i] == 0.0f) w[i >> 1] &= (i & 1) ? 0x0000FFFFu : 0xFFFF0000u;
            }
            store_codes8<FMT>(Q, r * C + c0, v, inv, false);
        }
    }
}

__global__ void rtne_col_scale_kernel(const uint32_t* bits, int64_t C, float* scale) {
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= C) return;
    const uint32_t m = bits[c];
    scale[c] = m >= 0x7F800000u ? __uint_as_float(0x7FC00000u) : (m ? __uint_as_float(m) / 127.0f : 1.0f);
}

}  // namespace s3r

using namespace s3r;

static bool valid_fmt(int fmt) { return fmt == S3R_CODES_S8 || fmt == S3R_CODES_F16; }

static PFN_cuTensorMapEncodeTiled_v12000 q_encode_fn() {
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

static int sm_count() { return s3r_sm_count(); }

int quant_wait_probe(uint64_t limit_ns, int* d_status, unsigned long long* waited_ns, cudaStream_t stream) {
    q_wait_probe_kernel<<<1, 32, 0, stream>>>(limit_ns, d_status, waited_ns);
    S3R_CHECK_LAUNCH();
    return S3R_OK;
}


template <int MODE, int FMT, bool FOLD>
static int launch_quant_tma(const CUtensorMap& map, const TileQuantArgs& A, const QuantCommon& C, const QuantOut& O,
                            int64_t ntiles, cudaStream_t stream) {
    const int st = s3r_kernel_smem((const void*)quantize_tma_kernel<MODE, FMT, FOLD>, kQuantTmaSmem,
                                   "quantize: cudaFuncSetAttribute");
    if (st) return st;
    const int64_t grid = ntiles < 2LL * sm_count() ? ntiles : 2LL * sm_count();
    quantize_tma_kernel<MODE, FMT, FOLD><<<(unsigned)grid, 256, kQuantTmaSmem, stream>>>(map, A, C, O, ntiles);
    S3R_CHECK_LAUNCH();
    return S3R_OK;
}

template <int MODE, int FMT>
static int launch_quant_tma(const CUtensorMap& map, const TileQuantArgs& A, const QuantCommon& C, const QuantOut& O,
                            int64_t ntiles, cudaStream_t stream) {
    return (A.s_x || A.s_w) ? launch_quant_tma<MODE, FMT, true>(map, A, C, O, ntiles, stream)
                            : launch_quant_tma<MODE, FMT, false>(map, A, C, O, ntiles, stream);
}

// The TMA path needs 16-byte aligned rows; returns 1 when it does not apply.
static int try_quant_tma(int mode, const TileQuantArgs& A, const QuantCommon& C, const QuantOut& O,
                         cudaStream_t stream) {
    if (!A.vec_load || !C.vec_store) return 1;
    auto fn = q_encode_fn();
    if (!fn) return 1;
    CUtensorMap map;
    cuuint64_t dims[2] = {(cuuint64_t)C.N, (cuuint64_t)C.T};
    cuuint64_t strides[1] = {(cuuint64_t)A.ldg * 2};
    cuuint32_t box[2] = {(cuuint32_t)kTile, (cuuint32_t)kTile};
    cuuint32_t estr[2] = {1u, 1u};
    if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(A.G), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return 1;
    const int64_t ntiles = s3r_cdiv(C.T, kTile) * C.ntc;
    if (ntiles >= (int64_t(1) << 31) / 4) return 1;   // the kernel keeps tile indices in 32 bits
    const bool f16 = O.fmt == S3R_CODES_F16;
    switch (mode) {
        case kRTNE: return f16 ? launch_quant_tma<kRTNE, 1>(map, A, C, O, ntiles, stream)
                               : launch_quant_tma<kRTNE, 0>(map, A, C, O, ntiles, stream);
        case kS3R: return f16 ? launch_quant_tma<kS3R, 1>(map, A, C, O, ntiles, stream)
                              : launch_quant_tma<kS3R, 0>(map, A, C, O, ntiles, stream);
        case kS3R7: return f16 ? launch_quant_tma<kS3R7, 1>(map, A, C, O, ntiles, stream)
                               : launch_quant_tma<kS3R7, 0>(map, A, C, O, ntiles, stream);
        case kBCAST: return f16 ? launch_quant_tma<kBCAST, 1>(map, A, C, O, ntiles, stream)
                                : launch_quant_tma<kBCAST, 0>(map, A, C, O, ntiles, stream);
        default: return f16 ? launch_quant_tma<kINDEP, 1>(map, A, C, O, ntiles, stream)
                            : launch_quant_tma<kINDEP, 0>(map, A, C, O, ntiles, stream);
    }
}

// Per-tensor step: max |g| of the folded gradient over the whole tensor, as a
// bit pattern (non-negative floats and NaN order like their bits), combined
// across CTAs with an atomic max (order-independent, so deterministic).
__global__ void __launch_bounds__(256) tensor_absmax_kernel(const uint16_t* G, int64_t T, int64_t N, int64_t ldg,
                                                            const float* s_x, const float* s_w, uint32_t* amax) {
    __shared__ uint32_t red[8];
    uint32_t m = 0u;
    const int64_t total = T * N;
    for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < total; i += (int64_t)gridDim.x * 256) {
        const int64_t t = i / N, n = i - t * N;
        float g = __uint_as_float((uint32_t)G[t * ldg + n] << 16);
        if (s_x) g = __fmul_rn(s_x[t], g);
        if (s_w) g = __fmul_rn(g, s_w[n]);
        m = max(m, __float_as_uint(g) & 0x7FFFFFFFu);
    }
    m = block_max_u32<8>(m, red);
    if (threadIdx.x == 0) atomicMax(amax, m);
}

// S: tokens per example (Phi_bcast; 0: one example).  tensor_amax: per-tensor
// step (a device float that receives max |g|), or null for one step per tile.
static int launch_tile_quant(int mode, const void* G, int64_t T, int64_t N, int64_t ldg, const float* s_x,
                             const float* s_w, uint64_t seed, uint32_t tensor_id, void* Q, int fmt, float* scale,
                             float* tok, float* col, int* d_status, cudaStream_t stream, int64_t S = 0,
                             float* tensor_amax = nullptr) {
    if (T < 0 || N < 0 || !valid_fmt(fmt) || S < 0) return S3R_ERR_ARG;
    if (T == 0 || N == 0) return S3R_OK;
    if (!G || !Q || !scale) return S3R_ERR_ARG;
    if (ldg < N) return S3R_ERR_SHAPE;
    if (s3r_cdiv(T, kTile) > 65535) return S3R_ERR_UNSUPPORTED;
    TileQuantArgs A{static_cast<const uint16_t*>(G), ldg, s_x, s_w, s3r_aligned16(G) && (ldg % 8) == 0};
    QuantCommon C{T, N, s3r_cdiv(N, kTile), (uint32_t)seed, d_status, s3r_aligned16(Q) && (N % 8) == 0, S,
                  reinterpret_cast<const uint32_t*>(tensor_amax)};
    QuantOut O{Q, fmt, scale, tok, col, tensor_id};
    if (tensor_amax) {
        cudaError_t e = cudaMemsetAsync(tensor_amax, 0, sizeof(float), stream);
        if (e != cudaSuccess) return s3r_cuda_fail("quantize: cudaMemsetAsync", e);
        const int64_t blocks = std::min<int64_t>(s3r_cdiv(T * N, 256), 8LL * sm_count());
        tensor_absmax_kernel<<<(unsigned)blocks, 256, 0, stream>>>(A.G, T, N, ldg, s_x, s_w,
                                                                   reinterpret_cast<uint32_t*>(tensor_amax));
        S3R_CHECK_LAUNCH();
    }
    const int tma = try_quant_tma(mode, A, C, O, stream);
    if (tma <= 0) return tma;   // launched (0) or failed (< 0)
    dim3 grid((unsigned)s3r_cdiv(N, kTile), (unsigned)s3r_cdiv(T, kTile));
    switch (mode) {
        case kRTNE: quantize_tile_kernel<kRTNE><<<grid, 256, 0, stream>>>(A, C, O); break;
        case kS3R: quantize_tile_kernel<kS3R><<<grid, 256, 0, stream>>>(A, C, O); break;
        case kINDEP: quantize_tile_kernel<kINDEP><<<grid, 256, 0, stream>>>(A, C, O); break;
        case kS3R7: quantize_tile_kernel<kS3R7><<<grid, 256, 0, stream>>>(A, C, O); break;
        case kBCAST: quantize_tile_kernel<kBCAST><<<grid, 256, 0, stream>>>(A, C, O); break;
        default: return S3R_ERR_ARG;
    }
    S3R_CHECK_LAUNCH();
    return S3R_OK;
}

extern "C" int s3r_quantize(const void* G, int64_t T, int64_t N, int64_t ldg, const float* s_x, const float* s_w,
                            uint64_t seed, uint32_t tensor_id, void* Q, int code_format, float* tile_scale,
                            float* tok_err_part, float* col_err_part, int* d_status, cudaStream_t stream) {
    return launch_tile_quant(kS3R, G, T, N, ldg, s_x, s_w, seed, tensor_id, Q, code_format, tile_scale, tok_err_part,
                             col_err_part, d_status, stream);
}

extern "C" int s3r_quantize_ex(const void* G, int64_t T, int64_t N, int64_t ldg, const float* s_x,
                               const float* s_w, int round_mode, int64_t S, float* tensor_amax, uint64_t seed,
                               uint32_t tensor_id, void* Q, int code_format, float* tile_scale, float* tok_err_part,
                               float* col_err_part, int* d_status, cudaStream_t stream) {
    int mode;
    switch (round_mode) {
        case S3R_ROUND_S3R: mode = kS3R; break;
        case S3R_ROUND_S3R_7BIT: mode = kS3R7; break;
        case S3R_ROUND_BCAST: mode = kBCAST; break;
        case S3R_ROUND_RTNE: mode = kRTNE; break;
        case S3R_ROUND_INDEP: mode = kINDEP; break;
        default: return S3R_ERR_ARG;
    }
    if (round_mode == S3R_ROUND_BCAST && S > 0 && T % S != 0) return S3R_ERR_SHAPE;
    const bool partials = round_mode == S3R_ROUND_S3R || round_mode == S3R_ROUND_S3R_7BIT ||
                          round_mode == S3R_ROUND_BCAST;
    return launch_tile_quant(mode, G, T, N, ldg, s_x, s_w, seed, tensor_id, Q, code_format, tile_scale,
                             partials ? tok_err_part : nullptr, partials ? col_err_part : nullptr, d_status, stream,
                             S, tensor_amax);
}

extern "C" int indep_sr_quantize(const void* G, int64_t T, int64_t N, int64_t ldg, const float* s_x,
                                 const float* s_w, uint64_t seed, uint32_t tensor_id, void* Q, int code_format,
                                 float* tile_scale, int* d_status, cudaStream_t stream) {
    return launch_tile_quant(kINDEP, G, T, N, ldg, s_x, s_w, seed, tensor_id, Q, code_format, tile_scale, nullptr,
                             nullptr, d_status, stream);
}

extern "C" int rtne_quantize(const void* A, int64_t R, int64_t C, int64_t lda, const float* s_x, const float* s_w,
                             int scale_axis, void* Q, int code_format, float* scale, int* d_status,
                             cudaStream_t stream) {
    if (scale_axis == S3R_AXIS_TILE)
        return launch_tile_quant(kRTNE, A, R, C, lda, s_x, s_w, 0, 0, Q, code_format, scale, nullptr, nullptr,
                                 d_status, stream);
    if (R < 0 || C < 0 || !valid_fmt(code_format)) return S3R_ERR_ARG;
    if (R == 0 || C == 0) return S3R_OK;
    if (!A || !Q || !scale) return S3R_ERR_ARG;
    if (lda < C) return S3R_ERR_SHAPE;
    if (s_x || s_w) return S3R_ERR_ARG;  // forward operands are not folded
    const uint16_t* a = static_cast<const uint16_t*>(A);
    const bool vec = s3r_aligned16(A) && s3r_aligned16(Q) && C % 8 == 0 && lda % 8 == 0;
    const bool f16 = code_format == S3R_CODES_F16;
    if (vec && scale_axis == S3R_AXIS_ROW && R <= 0x7FFFFFFF) {
        const unsigned nt = row_block_threads(C / 8);
        if (f16) rtne_rows_vec_kernel<S3R_CODES_F16><<<(unsigned)R, nt, 0, stream>>>(a, C, lda, Q, scale, d_status);
        else rtne_rows_vec_kernel<S3R_CODES_S8><<<(unsigned)R, nt, 0, stream>>>(a, C, lda, Q, scale, d_status);
        S3R_CHECK_LAUNCH();
        return S3R_OK;
    }
    if (vec && scale_axis == S3R_AXIS_COL && s3r_cdiv(R, kColChunk) <= 65535) {
        // the column maxima are gathered in `scale` itself (as bit patterns), then converted
        uint32_t* bits = reinterpret_cast<uint32_t*>(scale);
        const cudaError_t e = cudaMemsetAsync(bits, 0, (size_t)C * 4, stream);
        if (e != cudaSuccess) return s3r_cuda_fail("rtne_quantize: cudaMemsetAsync", e);
        const dim3 grid((unsigned)s3r_cdiv(C, kColStrip), (unsigned)s3r_cdiv(R, kColChunk));
        rtne_colmax_kernel<<<grid, 256, 0, stream>>>(a, R, C, lda, bits);
        S3R_CHECK_LAUNCH();
        if (f16) rtne_cols_vec_kernel<S3R_CODES_F16><<<grid, 256, 0, stream>>>(a, R, C, lda, Q, bits, d_status);
        else rtne_cols_vec_kernel<S3R_CODES_S8><<<grid, 256, 0, stream>>>(a, R, C, lda, Q, bits, d_status);
        S3R_CHECK_LAUNCH();
        rtne_col_scale_kernel<<<(unsigned)s3r_cdiv(C, 256), 256, 0, stream>>>(bits, C, scale);
        S3R_CHECK_LAUNCH();
        return S3R_OK;
    }
    if (scale_axis == S3R_AXIS_ROW) {
        if (R > 0x7FFFFFFF) return S3R_ERR_UNSUPPORTED;
        rtne_rows_kernel<<<(unsigned)R, 256, 0, stream>>>(a, R, C, lda, Q, code_format, scale, d_status);
    } else if (scale_axis == S3R_AXIS_COL) {
        rtne_cols_kernel<<<(unsigned)s3r_cdiv(C, 256), 256, 0, stream>>>(a, R, C, lda, Q, code_format, scale,
                                                                          d_status);
    } else {
        return S3R_ERR_ARG;
    }
    S3R_CHECK_LAUNCH();
    return S3R_OK;
}

extern "C" int swiglu_fwd_quantize(const void* h1, const void* h3, int64_t T, int64_t F, int64_t ldh, void* a,
                                   void* Q, int code_format, float* scale, int* d_status, cudaStream_t stream) {
    if (T < 0 || F < 0 || !valid_fmt(code_format)) return S3R_ERR_ARG;
    if (T == 0 || F == 0) return S3R_OK;
    if (!h1 || !h3 || !Q || !scale) return S3R_ERR_ARG;
    if (ldh < F) return S3R_ERR_SHAPE;
    if (T > 0x7FFFFFFF) return S3R_ERR_UNSUPPORTED;
    if (F % 8 != 0 || ldh % 8 != 0 || !s3r_aligned16(h1) || !s3r_aligned16(h3) || !s3r_aligned16(Q) ||
        (a && !s3r_aligned16(a)))
        return S3R_ERR_ALIGN;
    const uint16_t* p1 = static_cast<const uint16_t*>(h1);
    const uint16_t* p3 = static_cast<const uint16_t*>(h3);
    uint16_t* pa = static_cast<uint16_t*>(a);
    const unsigned nt = row_block_threads(F / 8);
    if (code_format == S3R_CODES_F16)
        swiglu_fwd_rows_kernel<S3R_CODES_F16><<<(unsigned)T, nt, 0, stream>>>(p1, p3, F, ldh, pa, Q, scale, d_status);
    else
        swiglu_fwd_rows_kernel<S3R_CODES_S8><<<(unsigned)T, nt, 0, stream>>>(p1, p3, F, ldh, pa, Q, scale, d_status);
    S3R_CHECK_LAUNCH();
    return S3R_OK;
}

template <int MODE, int FMT>
static int launch_swiglu_tma(const CUtensorMap* maps, const SwigluArgs& A, const QuantCommon& C, const QuantOut& O1,
                             const QuantOut& O3, int64_t ntiles, cudaStream_t stream) {
    const int st = s3r_kernel_smem((const void*)swiglu_tma_kernel<MODE, FMT>, kSwigluTmaSmem,
                                   "swiglu_quantize: cudaFuncSetAttribute");
    if (st) return st;
    const int64_t grid = ntiles < sm_count() ? ntiles : sm_count();
    swiglu_tma_kernel<MODE, FMT><<<(unsigned)grid, 512, kSwigluTmaSmem, stream>>>(maps[0], maps[1], maps[2], A, C,
                                                                                   O1, O3, ntiles);
    S3R_CHECK_LAUNCH();
    return S3R_OK;
}

// The TMA path needs 16-byte aligned rows (and codes); returns 1 when it does not apply.
static int try_swiglu_tma(int round_mode, const SwigluArgs& A, const QuantCommon& C, const QuantOut& O1,
                          const QuantOut& O3, cudaStream_t stream) {
    if (!A.vec_load || !C.vec_store) return 1;
    auto fn = q_encode_fn();
    if (!fn) return 1;
    CUtensorMap maps[3];
    cuuint64_t dims[2] = {(cuuint64_t)C.N, (cuuint64_t)C.T};
    cuuint32_t box[2] = {(cuuint32_t)kTile, (cuuint32_t)kSwQuarterRows};
    cuuint32_t estr[2] = {1u, 1u};
    cuuint64_t sd[1] = {(cuuint64_t)A.ldd * 4}, sh[1] = {(cuuint64_t)A.ldh * 2};
    if (fn(&maps[0], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(A.dA), dims, sd, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        fn(&maps[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(A.h1), dims, sh, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        fn(&maps[2], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(A.h3), dims, sh, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return 1;
    const int64_t ntiles = s3r_cdiv(C.T, kTile) * C.ntc;
    if (ntiles >= (int64_t(1) << 31) / 4) return 1;   // the kernel keeps quarter indices in 32 bits
    const bool f16 = O1.fmt == S3R_CODES_F16;
    if (O3.fmt != O1.fmt) return 1;
    switch (round_mode) {
        case S3R_ROUND_RTNE: return f16 ? launch_swiglu_tma<kRTNE, 1>(maps, A, C, O1, O3, ntiles, stream)
                                        : launch_swiglu_tma<kRTNE, 0>(maps, A, C, O1, O3, ntiles, stream);
        case S3R_ROUND_S3R: return f16 ? launch_swiglu_tma<kS3R, 1>(maps, A, C, O1, O3, ntiles, stream)
                                       : launch_swiglu_tma<kS3R, 0>(maps, A, C, O1, O3, ntiles, stream);
        case S3R_ROUND_S3R_7BIT: return f16 ? launch_swiglu_tma<kS3R7, 1>(maps, A, C, O1, O3, ntiles, stream)
                                            : launch_swiglu_tma<kS3R7, 0>(maps, A, C, O1, O3, ntiles, stream);
        case S3R_ROUND_BCAST: return f16 ? launch_swiglu_tma<kBCAST, 1>(maps, A, C, O1, O3, ntiles, stream)
                                         : launch_swiglu_tma<kBCAST, 0>(maps, A, C, O1, O3, ntiles, stream);
        case S3R_ROUND_INDEP: return f16 ? launch_swiglu_tma<kINDEP, 1>(maps, A, C, O1, O3, ntiles, stream)
                                         : launch_swiglu_tma<kINDEP, 0>(maps, A, C, O1, O3, ntiles, stream);
        default: return S3R_ERR_ARG;
    }
}

extern "C" int swiglu_quantize(const float* dA, int64_t ldd, const void* h1, const void* h3, int64_t ldh, int64_t T,
                               int64_t F, const float* s_x, const float* s_w1, const float* s_w3, int round_mode,
                               int code_format, uint64_t seed, uint32_t tid1, uint32_t tid3, void* Q1, float* scale1,
                               float* tok1, float* col1, void* Q3, float* scale3, float* tok3, float* col3,
                               int* d_status, cudaStream_t stream) {
    return swiglu_quantize_ex(dA, ldd, h1, h3, ldh, T, F, s_x, s_w1, s_w3, round_mode, 0, code_format, seed, tid1,
                              tid3, Q1, scale1, tok1, col1, Q3, scale3, tok3, col3, d_status, stream);
}

extern "C" int swiglu_quantize_ex(const float* dA, int64_t ldd, const void* h1, const void* h3, int64_t ldh,
                                  int64_t T, int64_t F, const float* s_x, const float* s_w1, const float* s_w3,
                                  int round_mode, int64_t S, int code_format, uint64_t seed, uint32_t tid1,
                                  uint32_t tid3, void* Q1, float* scale1, float* tok1, float* col1, void* Q3,
                                  float* scale3, float* tok3, float* col3, int* d_status, cudaStream_t stream) {
    if (T < 0 || F < 0 || !valid_fmt(code_format) || S < 0) return S3R_ERR_ARG;
    if (round_mode == S3R_ROUND_BCAST && S > 0 && T % S != 0) return S3R_ERR_SHAPE;
    if (T == 0 || F == 0) return S3R_OK;
    if (!dA || !h1 || !h3 || !Q1 || !Q3 || !scale1 || !scale3) return S3R_ERR_ARG;
    if (ldd < F || ldh < F) return S3R_ERR_SHAPE;
    if (s3r_cdiv(T, kTile) > 65535) return S3R_ERR_UNSUPPORTED;
    SwigluArgs A{dA, ldd, static_cast<const uint16_t*>(h1), static_cast<const uint16_t*>(h3), ldh, s_x, s_w1, s_w3,
                 s3r_aligned16(dA) && s3r_aligned16(h1) && s3r_aligned16(h3) && (ldd % 4) == 0 && (ldh % 8) == 0};
    QuantCommon C{T, F, s3r_cdiv(F, kTile), (uint32_t)seed, d_status,
                  s3r_aligned16(Q1) && s3r_aligned16(Q3) && (F % 8) == 0, S, nullptr};
    QuantOut O1{Q1, code_format, scale1, tok1, col1, tid1}, O3{Q3, code_format, scale3, tok3, col3, tid3};
    const int tma = try_swiglu_tma(round_mode, A, C, O1, O3, stream);
    if (tma <= 0) return tma;   // launched (0) or failed (< 0)
    dim3 grid((unsigned)s3r_cdiv(F, kTile), (unsigned)s3r_cdiv(T, kTile));
    switch (round_mode) {
        case S3R_ROUND_RTNE: swiglu_quantize_kernel<kRTNE><<<grid, 512, 0, stream>>>(A, C, O1, O3); break;
        case S3R_ROUND_S3R: swiglu_quantize_kernel<kS3R><<<grid, 512, 0, stream>>>(A, C, O1, O3); break;
        case S3R_ROUND_S3R_7BIT: swiglu_quantize_kernel<kS3R7><<<grid, 512, 0, stream>>>(A, C, O1, O3); break;
        case S3R_ROUND_BCAST: swiglu_quantize_kernel<kBCAST><<<grid, 512, 0, stream>>>(A, C, O1, O3); break;
        case S3R_ROUND_INDEP: swiglu_quantize_kernel<kINDEP><<<grid, 512, 0, stream>>>(A, C, O1, O3); break;
        default: return S3R_ERR_ARG;
    }
    S3R_CHECK_LAUNCH();
    return S3R_OK;
}

// ---------------------------------------------------------------------------
// Test hook: the glue's reciprocal against the IEEE one over a range of bit
// patterns (grid-stride, one atomic per thread with a mismatch).
// ---------------------------------------------------------------------------
namespace {
__global__ void __launch_bounds__(256) check_reciprocal_kernel(uint32_t lo, uint32_t hi, unsigned long long* count) {
    const uint64_t n = (uint64_t)(hi - lo);
    unsigned long long bad = 0;
    for (uint64_t i = 2 * ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x); i < n;
         i += 2 * (uint64_t)gridDim.x * blockDim.x) {
        const float a = __uint_as_float(lo + (uint32_t)i);
        const float b = i + 1 < n ? __uint_as_float(lo + (uint32_t)i + 1) : a;
        const float2 r = s3r::rcp2_den(make_float2(a, b));
        bad += __float_as_uint(r.x) != __float_as_uint(__frcp_rn(a));
        bad += __float_as_uint(r.y) != __float_as_uint(__frcp_rn(b));
    }
    if (bad) atomicAdd(count, bad);
}
}  // namespace

extern "C" int s3r_check_reciprocal(uint32_t lo_bits, uint32_t hi_bits, unsigned long long* d_count,
                                    cudaStream_t stream) {
    if (!d_count || lo_bits >= hi_bits || hi_bits > 0x7F800000u || lo_bits == 0u) return S3R_ERR_ARG;
    const int grid = s3r_sm_count() * 8;
    check_reciprocal_kernel<<<grid, 256, 0, stream>>>(lo_bits, hi_bits, d_count);
    S3R_CHECK_LAUNCH();
    return S3R_OK;
}
