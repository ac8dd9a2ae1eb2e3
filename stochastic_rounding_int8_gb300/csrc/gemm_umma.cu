// gemm_umma.cu -- the INT8 GEMMs on the 5th-generation tensor cores (tcgen05,
// sm_103a), with the codes carried exactly in fp16: the backward's dX and dW
// (per-block promotion, correction in the epilogue) and, in a kernel
// instantiation of their own, the forward's Y = X W and gate/up projections
// (exact integer accumulation, see kFwdUnit).
//
// Paper: "Efficient Quantization Training with Stochastic Rounding via
// Structured Subspace Randomness" §III-A: S8 x S8 GEMM with S32 accumulation,
// then rescale; §III-D: subtract the image of the error projection.
//
// sm_103a has no integer tcgen05 MMA, and the warp-level s8 mma.sync path
// runs far below the 16-bit tensor rate on this part.  Every code is an
// integer in [-127, 127], exact in fp16, and a 128-long block of products is
// bounded by 128 * 127^2 < 2^24, so kind::f16 with an fp32 accumulator yields
// the exact int32 block sum.  The accumulator is drained after every 128-wide
// contraction block and promoted with that block's scale, as the per-tile
// quantization requires.
//
// Kernel layout: persistent, one CTA per SM looping over 128 x 256 output
// tiles (N fastest); 384 threads in three warpgroups:
//   warp 0      TMA producer: 4-stage ring of 64-deep K slices in smem
//               (128-byte swizzle), one mbarrier pair per stage;
//   warp 1      allocates 512 TMEM columns; lane 0 issues tcgen05.mma
//               (M=128, N=256, K=16) into one of two 256-column fp32
//               accumulators (double buffer) and commits to mbarriers;
//   warps 2, 3  idle (they complete warpgroup 0 for the register split);
//   warps 4..11 epilogue: per 128-K block, tcgen05.ld their 32 TMEM lanes x
//               128 columns, acc = fma(scale, block, acc) in registers (acc
//               seeded with minus the correction); at the end of the tile the
//               1/s rescale and coalesced fp32 stores, while the producer and
//               the MMA issuer already run the next tile.
// Warpgroup 0 gives registers to the epilogue warpgroups (setmaxnreg), so a
// drain keeps four TMEM loads in flight next to the 128 accumulators.
// The activation gradient may contract two operand pairs into one
// accumulator (dX = Q1 W1^T + Q3 W3^T), each with its own scales.
// Every mbarrier wait is bounded (S3R_ERR_TIMEOUT in d_status, clean exit).
#include <cstdio>
#include <algorithm>
#include <atomic>
#include <cstring>
#include <vector>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace s3r {
namespace umma {

constexpr int BM = 128, BN = 256, BKS = 64, STAGES = 4;
constexpr int A_STAGE = BM * BKS * 2;       // 16 KiB
constexpr int B_STAGE = BN * BKS * 2;       // 32 KiB
constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
constexpr int MN_ATOM_BYTES = BKS * 128;    // one 64-wide MN atom column over a 64-deep K slice: 8 KiB
constexpr int THREADS = 384;               // three warpgroups
constexpr int EPI_WARP0 = 4;                // epilogue warps 4..11 (warpgroups 1 and 2)
// Register split (setmaxnreg): warpgroup 0 (producer, MMA issuer, two idle
// warps) drops to kRegsLow, the epilogue warpgroups rise to kRegsHigh.  The
// launch holds regs_per_thread * 384 registers; the split needs
// kRegsLow * 128 + kRegsHigh * 256 of them, so the host refuses to launch a
// build whose per-thread count is below kMinLaunchRegs (an increase that the
// pool cannot satisfy would wait forever).
constexpr int kRegsLow = 40, kRegsHigh = 216;
constexpr int kMinLaunchRegs = (kRegsLow * 128 + kRegsHigh * 256 + 383) / 384;
constexpr int EPI_WARPS = 8;
constexpr int CHUNK = 16;                   // columns per epilogue staging round
constexpr int STAGE_PITCH = 20;             // floats per staged row: conflict-free 16-byte writes
constexpr int EPI_STAGE_BYTES = EPI_WARPS * 32 * STAGE_PITCH * 4;   // 20 KiB
constexpr int kNbX = 4;                     // dX: examples one 128-row tile may span (S >= 43)
constexpr int kBch = 8;                     // dW: examples staged per pass
constexpr int CV_FLOATS = 256 + 2 * kNbX * 128;   // per half; the dW layout (128 + kBch * 128) fits too
static_assert(128 + kBch * 128 <= CV_FLOATS, "dW column staging fits the dX layout's size");
constexpr int CV_BYTES = 2 * CV_FLOATS * 4;        // 10 KiB
constexpr uint32_t TMEM_COLS = 512;
constexpr int NUM_BARS = 2 * STAGES + 5;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_STAGE_BYTES + CV_BYTES + 1024 + NUM_BARS * 8 + 16;
static_assert(SMEM_BYTES + 64 <= 232448, "shared memory budget of one sm_103a CTA");
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait

// Epilogue kinds; a kMixed launch takes each problem's kind (kDX or kDW) from
// the problem, a kFwdE launch (forward problems only) too (kFwd or kGate).
// The forward gets its own instantiation so that the backward kernels carry
// none of its code.
enum Epi { kDX = 0, kDW = 1, kDump = 2, kMixed = 3, kFwdE = 4 };
// Problem kind of the INT8 forward (mixed launches only): A = X [M, K] K-major,
// B = W [K, N] MN-major, unit block scales, epilogue (acc * s_x[m]) * s_w[n].
constexpr int kFwd = 4;
// Problem kind of the gate and up projections with the SwiGLU gate in the
// epilogue (mixed launches only): one 128-column slice of W1 and the same
// slice of W3 fill the 256 accumulator columns, and the epilogue writes
// h1 = bf16(s_x s_w1 X W1), h3 = bf16(s_x s_w3 X W3) and a = bf16(silu(h1) h3).
constexpr int kGate = 5;
// Forward problems have unit block scales, so their accumulator is drained once
// per kFwdUnit 128-wide blocks: the TMEM partial over 1024 products of codes is
// below 1024 * 127^2 < 2^24 in magnitude, an exact integer in fp32; the
// epilogue adds the units as int32 (the exact S32 sum) and converts once.
constexpr int kFwdUnit = 8;

// One contraction segment: scale(mt, nt, kb) = scale[mt*sm + nt*sn + kb*sk],
// and for the activation gradient its correction terms.
struct Segment {
    const float* scale;
    int64_t sm, sn, sk, nt_limit;
    int64_t K;                   // contraction length of this segment
    const float* eps;
    const int32_t* rowsum;
    const float* v;
};

// One GEMM of a launch: C[M, N] = sum over segments of sum_k A[m, k] B[n, k],
// promoted per 128-wide block, corrected and rescaled in the epilogue.
struct Problem {
    int64_t M, N;
    int kind;                    // kDX (K-major operands) or kDW (MN-major operands)
    int ntm, ntn;                // 128 x 256 tiles along M and N
    int tile_base;               // first tile of this problem in the launch's tile order
    int band_rows;               // tile order inside the problem (tile_coords)
    Segment seg[2];              // seg[1].K == 0 when there is one segment
    float* C;
    int64_t ldc;
    int32_t* dump;
    const float* s_row;          // dX: 1/s_x[row] rescale
    const float* s_col;          // dW: 1/s_w[col] rescale
    const float* f_row;          // forward: s_x[row] multiplier (then f_col[col])
    const float* f_col;
    const float* f_col3;         // gate: s_w3
    uint16_t* gate_out[3];       // gate: h1, h3, a (bf16, row stride ldc)
    int ec_mode;
    int64_t S, B;
    const float* colmean;
    const float* mu;
    const int32_t* xsum;
    const float* p;
    int accumulate;
};

// A launch: up to kMaxProb problems (of one kind, or mixed), their tiles numbered one
// after another; each problem has up to four tensor maps (A and B of each
// segment).  Both live in the constant parameter space (__grid_constant__),
// so indexing them with a run-time problem number costs no copy.
constexpr int kMaxProb = 24;
struct Args {
    Problem prob[kMaxProb];
    int nprob;
    int total_tiles;
    int* d_status;
};
struct Maps {
    CUtensorMap m[kMaxProb][4];
};

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t gtime() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for the phase of the given parity to complete; gives up (false) after
// kWaitNs or as soon as another role raised the abort flag.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = gtime();
    while (!mbar_try(bar, parity)) {
        if (*abort_flag) return false;
        if (gtime() - t0 > kWaitNs) return false;
    }
    return true;
}
// Bounded wait that ignores the abort flag: used before teardown, where the
// copies or MMAs still in flight must land whatever the other roles did.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = gtime();
    while (!mbar_try(bar, parity))
        if (gtime() - t0 > kWaitNs) return false;
    return true;
}

__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"((uint64_t)map), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// Shared-memory matrix descriptor (tcgen05): start address, leading / stride
// byte offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor for kind::f16: fp32 accumulate, fp16 A and B,
// operand majorness, N >> 3 and M >> 4.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
            d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accum));
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 TMEM lanes x 16 consecutive 32-bit columns: thread i gets lane (base + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Per-tile column vectors, staged in shared memory by the four epilogue warps
// of each 128-column half (one column per thread, coalesced), so that the
// per-thread seed and rescale below are branch-free broadcast smem reads:
//   dX: rowsum_g[128] for g < 2, then v_g[b_lo + i][128] for i < kNbX;
//   dW: 1/s_w[128], then colmean[b][128] - mu[b] for a chunk of kBch examples.
// Columns past N are staged as 0.
__device__ __forceinline__ void half_bar(int half) {
    asm volatile("bar.sync %0, %1;" ::"r"(1 + half), "r"(128) : "memory");
}

__device__ __forceinline__ float4 lds4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// Seeds the thread's 128 accumulators (row `row`, columns c0..c0+127) with
// minus the correction, which does not depend on the contraction:
//   dX: -(eps_g[t] rowsum_g[k] + v_g[t/S, k]) summed over the terms g;
//   dW: -(p[k] + sum_b xsum[b, k] (colmean[b, n] - mu[b])).
// The dW pass also stages 1/s_w for the final rescale.
template <int EPI>
__device__ __forceinline__ void seed_tile(const Problem& P, float (&acc)[128], float* cv, int64_t row, int64_t m0,
                                          int64_t c0, int half, int ht) {
    const bool in = row < P.M;
    const int64_t cc = c0 + ht;   // the column this thread stages
    const bool cin = cc < P.N;
    if (EPI == kDX) {
        if (!P.ec_mode) {
#pragma unroll
            for (int j = 0; j < 128; ++j) acc[j] = 0.0f;
            return;
        }
        const int64_t b_lo = m0 / P.S;
        const int64_t b_hi = ((m0 + BM - 1 < P.M ? m0 + BM - 1 : P.M - 1)) / P.S;
        half_bar(half);   // every thread of the half is past its previous use of cv
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            const bool on = g == 0 || P.seg[1].K > 0;
            cv[g * 128 + ht] = (on && cin) ? (float)__ldg(P.seg[g].rowsum + cc) : 0.0f;
            for (int i = 0; i < kNbX; ++i)   // staged negated: the seed below is one fma per pair
                cv[256 + (g * kNbX + i) * 128 + ht] =
                    (on && cin && b_lo + i <= b_hi) ? -__ldg(P.seg[g].v + (b_lo + i) * P.N + cc) : 0.0f;
        }
        half_bar(half);
        const float ep0 = in ? __ldg(P.seg[0].eps + row) : 0.0f;
        const float ep1 = (in && P.seg[1].K > 0) ? __ldg(P.seg[1].eps + row) : 0.0f;
        const int i_row = in ? (int)(row / P.S - b_lo) : 0;
        // -(ep rowsum + v) = fma(-ep, rowsum, -v) exactly (v is staged negated)
        const float* rs0 = cv;
        const float* nv0 = cv + 256 + i_row * 128;
        const float2 nep0 = make_float2(-ep0, -ep0);
#pragma unroll
        for (int j4 = 0; j4 < 128; j4 += 4) {
            const float4 r = lds4(rs0 + j4), w = lds4(nv0 + j4);
            const float2 a = f2_fma(nep0, make_float2(r.x, r.y), make_float2(w.x, w.y));
            const float2 b = f2_fma(nep0, make_float2(r.z, r.w), make_float2(w.z, w.w));
            acc[j4 + 0] = a.x;
            acc[j4 + 1] = a.y;
            acc[j4 + 2] = b.x;
            acc[j4 + 3] = b.y;
        }
        if (P.seg[1].K > 0) {
            const float* rs1 = cv + 128;
            const float* nv1 = cv + 256 + (kNbX + i_row) * 128;
            const float2 nep1 = make_float2(-ep1, -ep1);
#pragma unroll
            for (int j4 = 0; j4 < 128; j4 += 4) {
                const float4 r = lds4(rs1 + j4), w = lds4(nv1 + j4);
                const float2 a = f2_add(make_float2(acc[j4], acc[j4 + 1]),
                                        f2_fma(nep1, make_float2(r.x, r.y), make_float2(w.x, w.y)));
                const float2 b = f2_add(make_float2(acc[j4 + 2], acc[j4 + 3]),
                                        f2_fma(nep1, make_float2(r.z, r.w), make_float2(w.z, w.w)));
                acc[j4 + 0] = a.x;
                acc[j4 + 1] = a.y;
                acc[j4 + 2] = b.x;
                acc[j4 + 3] = b.y;
            }
        }
    } else {
        const bool two = P.ec_mode == S3R_EC_TWO_WAY;
        const float pr = (two && in) ? __ldg(P.p + row) : 0.0f;
#pragma unroll
        for (int j = 0; j < 128; ++j) acc[j] = pr;
        const int64_t nb = two ? P.B : 0;
        for (int64_t b0 = 0; b0 == 0 || b0 < nb; b0 += kBch) {
            half_bar(half);   // every thread of the half is past its previous use of cv
            if (b0 == 0) cv[ht] = (P.s_col && cin) ? __frcp_rn(__ldg(P.s_col + cc)) : 1.0f;
            for (int i = 0; i < kBch; ++i)
                cv[128 + i * 128 + ht] =
                    (cin && b0 + i < nb) ? __ldg(P.colmean + (b0 + i) * P.N + cc) - __ldg(P.mu + b0 + i) : 0.0f;
            half_bar(half);
            const int64_t nbi = nb - b0 < kBch ? nb - b0 : kBch;
            for (int64_t i = 0; i < nbi; ++i) {
                const float xs = in ? (float)__ldg(P.xsum + (b0 + i) * P.M + row) : 0.0f;
                const float* cm = cv + 128 + i * 128;
                const float2 xs2 = make_float2(xs, xs);
#pragma unroll
                for (int j4 = 0; j4 < 128; j4 += 4) {
                    const float4 c4 = lds4(cm + j4);
                    const float2 a = f2_fma(xs2, make_float2(c4.x, c4.y), make_float2(acc[j4], acc[j4 + 1]));
                    const float2 b = f2_fma(xs2, make_float2(c4.z, c4.w), make_float2(acc[j4 + 2], acc[j4 + 3]));
                    acc[j4 + 0] = a.x;
                    acc[j4 + 1] = a.y;
                    acc[j4 + 2] = b.x;
                    acc[j4 + 3] = b.y;
                }
            }
        }
#pragma unroll
        for (int j = 0; j < 128; ++j) acc[j] = -acc[j];
    }
}

// Final epilogue of one warp's 32 x 128 block (thread = row, acc = its 128
// columns from c0, already corrected): the rescale (times 1/s_x[t] or the
// staged 1/s_w[n]), then 16-column rounds through the warp's staging buffer
// so that every global access is a 64-byte row segment (accumulate reads
// included).
template <int EPI, bool FWD = false>
__device__ __forceinline__ void finish_tile(const Problem& P, float (&acc)[128], const float* cv, float* stage,
                                            int64_t row, int64_t c0, int lane) {
    if (FWD) {
        // forward: the exact int32 sum converted once, then (acc * s_x[row]) * s_w[col], one
        // rounding each, columns past N scaled by 1
#pragma unroll
        for (int j = 0; j < 128; ++j) acc[j] = __int2float_rn(__float_as_int(acc[j]));
        const float fr = row < P.M ? __ldg(P.f_row + row) : 1.0f;
        const float2 fr2 = make_float2(fr, fr);
        const bool fvec = (reinterpret_cast<uintptr_t>(P.f_col) & 15u) == 0;
#pragma unroll
        for (int j4 = 0; j4 < 128; j4 += 4) {
            const int64_t col = c0 + j4;
            const float4 fc = (fvec && col + 4 <= P.N)
                                  ? __ldg(reinterpret_cast<const float4*>(P.f_col + col))
                                  : make_float4(col < P.N ? __ldg(P.f_col + col) : 1.0f,
                                                col + 1 < P.N ? __ldg(P.f_col + col + 1) : 1.0f,
                                                col + 2 < P.N ? __ldg(P.f_col + col + 2) : 1.0f,
                                                col + 3 < P.N ? __ldg(P.f_col + col + 3) : 1.0f);
            const float2 a = f2_mul(f2_mul(make_float2(acc[j4], acc[j4 + 1]), fr2), make_float2(fc.x, fc.y));
            const float2 b = f2_mul(f2_mul(make_float2(acc[j4 + 2], acc[j4 + 3]), fr2), make_float2(fc.z, fc.w));
            acc[j4] = a.x;
            acc[j4 + 1] = a.y;
            acc[j4 + 2] = b.x;
            acc[j4 + 3] = b.y;
        }
    }
    if (EPI == kDX && P.s_row) {
        const float rinv = row < P.M ? __frcp_rn(__ldg(P.s_row + row)) : 1.0f;
        const float2 r2 = make_float2(rinv, rinv);
#pragma unroll
        for (int j = 0; j < 128; j += 2) {
            const float2 a = f2_mul(make_float2(acc[j], acc[j + 1]), r2);
            acc[j] = a.x;
            acc[j + 1] = a.y;
        }
    }
    if (EPI == kDW && P.s_col) {
#pragma unroll
        for (int j4 = 0; j4 < 128; j4 += 4) {
            const float4 r = lds4(cv + j4);
            const float2 a = f2_mul(make_float2(acc[j4], acc[j4 + 1]), make_float2(r.x, r.y));
            const float2 b = f2_mul(make_float2(acc[j4 + 2], acc[j4 + 3]), make_float2(r.z, r.w));
            acc[j4 + 0] = a.x;
            acc[j4 + 1] = a.y;
            acc[j4 + 2] = b.x;
            acc[j4 + 3] = b.y;
        }
    }
    const bool cvec = (P.ldc % 4 == 0) && ((reinterpret_cast<uintptr_t>(P.C) & 15u) == 0);
    const bool accum = EPI == kDX && P.accumulate;
    const int srow = lane >> 2, scol = 4 * (lane & 3);   // store mapping: 8 rows x 4 float4 per instruction
    const int64_t row0 = row - lane;
    float* mine = stage + lane * STAGE_PITCH;
#pragma unroll
    for (int c = 0; c < 128 / CHUNK; ++c) {
#pragma unroll
        for (int j4 = 0; j4 < CHUNK; j4 += 4)
            *reinterpret_cast<float4*>(mine + j4) = make_float4(acc[CHUNK * c + j4], acc[CHUNK * c + j4 + 1],
                                                                acc[CHUNK * c + j4 + 2], acc[CHUNK * c + j4 + 3]);
        __syncwarp();
        const int64_t col = c0 + CHUNK * c + scol;
#pragma unroll 1
        for (int r8 = 0; r8 < 4; ++r8) {
            const int lr = 8 * r8 + srow;
            const int64_t grow = row0 + lr;
            if (grow < P.M && col < P.N) {
                const float4 v4 = lds4(stage + lr * STAGE_PITCH + scol);
                float w[4] = {v4.x, v4.y, v4.z, v4.w};
                float* dst = P.C + grow * P.ldc + col;
                if (cvec && col + 4 <= P.N) {
                    if (accum) {
                        const float4 t = *reinterpret_cast<const float4*>(dst);
                        w[0] += t.x; w[1] += t.y; w[2] += t.z; w[3] += t.w;
                    }
                    *reinterpret_cast<float4*>(dst) = make_float4(w[0], w[1], w[2], w[3]);
                } else {
                    for (int j = 0; j < 4; ++j)
                        if (col + j < P.N) dst[j] = accum ? w[j] + dst[j] : w[j];
                }
            }
        }
        __syncwarp();
    }
}

// Gate epilogue of the forward (thread = row, acc[0..63] = h1 and acc[64..127]
// = h3 accumulators of output columns c0 .. c0 + 63, as exact int32 sums):
// convert to fp32 once, rescale in fp32 as (acc * s_x) * s_w and round to
// bf16 (nearest even).  With an `a` output the
// gate follows from those bf16 values: a = bf16((h1 * sigmoid(h1)) * h3).
// Each thread writes its row's 64 columns as 16-byte pieces; N is a multiple
// of 8, so a group of 8 columns lies wholly inside or outside.
__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&p);
}

__device__ __forceinline__ void finish_gate(const Problem& P, float (&acc)[128], int64_t row, int64_t c0) {
    if (row >= P.M) return;
#pragma unroll
    for (int j = 0; j < 128; ++j) acc[j] = __int2float_rn(__float_as_int(acc[j]));   // the exact int32 sums
    const float fr = __ldg(P.f_row + row);
    const float2 fr2 = make_float2(fr, fr);
    uint16_t* const out_a = P.gate_out[2];
    const bool vec = (P.ldc % 8 == 0) &&
                     ((reinterpret_cast<uintptr_t>(P.gate_out[0]) | reinterpret_cast<uintptr_t>(P.gate_out[1]) |
                       reinterpret_cast<uintptr_t>(out_a) | reinterpret_cast<uintptr_t>(P.f_col) |
                       reinterpret_cast<uintptr_t>(P.f_col3)) & 15u) == 0;
#pragma unroll
    for (int j8 = 0; j8 < 64; j8 += 8) {
        const int64_t col = c0 + j8;
        if (col >= P.N) break;
        float s1[8], s3[8];
        if (vec) {
            const float4* p1 = reinterpret_cast<const float4*>(P.f_col + col);
            const float4* p3 = reinterpret_cast<const float4*>(P.f_col3 + col);
            const float4 a0 = __ldg(p1), a1 = __ldg(p1 + 1), b0 = __ldg(p3), b1 = __ldg(p3 + 1);
            s1[0] = a0.x; s1[1] = a0.y; s1[2] = a0.z; s1[3] = a0.w; s1[4] = a1.x; s1[5] = a1.y; s1[6] = a1.z; s1[7] = a1.w;
            s3[0] = b0.x; s3[1] = b0.y; s3[2] = b0.z; s3[3] = b0.w; s3[4] = b1.x; s3[5] = b1.y; s3[6] = b1.z; s3[7] = b1.w;
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                s1[j] = __ldg(P.f_col + col + j);
                s3[j] = __ldg(P.f_col3 + col + j);
            }
        }
        uint32_t w1[4], w3[4], wa[4];
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            const float2 h1 = f2_mul(f2_mul(make_float2(acc[j8 + j], acc[j8 + j + 1]), fr2), make_float2(s1[j], s1[j + 1]));
            const float2 h3 =
                f2_mul(f2_mul(make_float2(acc[64 + j8 + j], acc[64 + j8 + j + 1]), fr2), make_float2(s3[j], s3[j + 1]));
            w1[j / 2] = bf16x2_bits(h1.x, h1.y);
            w3[j / 2] = bf16x2_bits(h3.x, h3.y);
        }
        const int64_t off = row * P.ldc + col;
        if (out_a) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 x = make_float2(__uint_as_float(w1[k] << 16), __uint_as_float(w1[k] & 0xFFFF0000u));
                const float2 z = make_float2(__uint_as_float(w3[k] << 16), __uint_as_float(w3[k] & 0xFFFF0000u));
                const float2 av = f2_mul(f2_mul(x, sigmoid2(x)), z);
                wa[k] = bf16x2_bits(av.x, av.y);
            }
        }
        if (vec) {
            *reinterpret_cast<uint4*>(P.gate_out[0] + off) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
            *reinterpret_cast<uint4*>(P.gate_out[1] + off) = make_uint4(w3[0], w3[1], w3[2], w3[3]);
            if (out_a) *reinterpret_cast<uint4*>(out_a + off) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int sh = 16 * (j & 1);
                P.gate_out[0][off + j] = (uint16_t)(w1[j / 2] >> sh);
                P.gate_out[1][off + j] = (uint16_t)(w3[j / 2] >> sh);
                if (out_a) out_a[off + j] = (uint16_t)(wa[j / 2] >> sh);
            }
        }
    }
}

// Tile order: bands of `band` row tiles; inside a band the row index runs
// fastest, then the column (band = 1 is plain column-fastest order).  The
// host picks the band height that makes the first wave of concurrent CTAs
// touch the fewest operand bytes (row strips of A plus column strips of B),
// so more of each wave's operands are shared in L2.
__host__ __device__ __forceinline__ void tile_coords(int tile, int ntm, int ntn, int band_rows, int& tm,
                                                     int& tn) {
    const int band = tile / (band_rows * ntn);
    const int rows = min(band_rows, ntm - band * band_rows);   // the last band may be thinner
    const int in = tile - band * band_rows * ntn;
    tm = band * band_rows + in % rows;
    tn = in / rows;
}

// The problem that owns launch tile `tile` (tiles of problem i start at
// prob[i].tile_base, in increasing order).
__device__ __forceinline__ int problem_of(const Args& A, int tile) {
    int i = 0;
    while (i + 1 < A.nprob && tile >= A.prob[i + 1].tile_base) ++i;
    return i;
}

// 12 warps: one SM sub-partition hosts three of them, one per warpgroup, so the
// launch is capped at 168 registers per thread; after the split a
// sub-partition holds (40 + 216 + 216) * 32 = 15104 of its 16384.
template <int EPI, bool MN>
__global__ void __launch_bounds__(THREADS, 1)
    umma_gemm_kernel(const __grid_constant__ Maps maps, const __grid_constant__ Args A) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ int abort_flag;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_STAGE;
    float* sEpi = reinterpret_cast<float*>(sB + STAGES * B_STAGE);
    float* sCv = sEpi + EPI_STAGE_BYTES / 4;
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sCv) + CV_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
    const uint32_t full0 = su32(bars), empty0 = su32(bars + STAGES), tfull0 = su32(bars + 2 * STAGES),
                   tempty0 = su32(bars + 2 * STAGES + 2), done_bar = su32(bars + 2 * STAGES + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntiles = A.total_tiles;   // tile counts fit 32 bits (checked by the host)

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8 * b, 1);
            mbar_init(tempty0 + 8 * b, EPI_WARPS);
        }
        mbar_init(done_bar, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tmem = *tmem_slot;
    volatile int* abrt = &abort_flag;

    // Persistent: this CTA owns tiles blockIdx.x, blockIdx.x + gridDim.x, ...;
    // tiles run along N first.  The smem ring and the TMEM double buffer keep
    // their phases across tiles, so the next tile's copies and MMAs start while
    // the epilogue still stores the previous tile.
    if (warp < EPI_WARP0) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
        if (warp == 0) {
            if (lane == 0) {
                int it = 0;   // slice counter over the whole persistent run
                int last_pi = -1;
                bool ok = true;
                for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                    const int pi = problem_of(A, tile);
                    const Problem& P = A.prob[pi];
                    const CUtensorMap* mp = &maps.m[pi][0];
                    const int nkb0 = (int)s3r_cdiv(P.seg[0].K, 128), nkb1 = (int)s3r_cdiv(P.seg[1].K, 128);
                    const int nkb = nkb0 + nkb1;   // 128-wide blocks of this tile
                    if (pi != last_pi) {
                        for (int j = 0; j < (nkb1 || (EPI == kFwdE && P.kind == kGate) ? 4 : 2); ++j)
                            asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)(mp + j)) : "memory");
                        last_pi = pi;
                    }
                    int tm, tn;
                    tile_coords(tile - P.tile_base, P.ntm, P.ntn, P.band_rows, tm, tn);
                    const bool gate = EPI == kFwdE && P.kind == kGate;
                    const int32_t m0 = tm * BM, n0 = tn * (gate ? BN / 2 : BN);
                    for (int sl = 0; sl < 2 * nkb; ++sl, ++it) {
                        const int s = it % STAGES;
                        if (!mbar_wait(empty0 + 8 * s, ((uint32_t)(it / STAGES) & 1u) ^ 1u, abrt)) {
                            *abrt = 1;
                            ok = false;
                            ++it;
                            break;
                        }
                        const uint32_t fb = full0 + 8 * s;
                        mbar_expect_tx(fb, STAGE_BYTES);
                        const bool second = sl >= 2 * nkb0;
                        const CUtensorMap* mA = mp + (second ? 2 : 0);
                        const CUtensorMap* mB = mp + (second ? 3 : 1);
                        const int32_t k0 = (second ? sl - 2 * nkb0 : sl) * BKS;
                        const uint32_t a_dst = su32(sA + s * A_STAGE), b_dst = su32(sB + s * B_STAGE);
                        // forward: A K-major, B MN-major as stored
                        const bool a_mn = EPI == kMixed ? P.kind == kDW : (EPI == kFwdE ? false : MN);
                        const bool b_mn = EPI == kMixed ? P.kind == kDW : (EPI == kFwdE ? true : MN);
                        if (!a_mn) {
                            tma_load(a_dst, mA, k0, m0, fb);
                        } else {
                            tma_load(a_dst, mA, m0, k0, fb);
                            tma_load(a_dst + MN_ATOM_BYTES, mA, m0 + 64, k0, fb);
                        }
                        if (!b_mn) {
                            tma_load(b_dst, mB, k0, n0, fb);
                        } else {
#pragma unroll
                            for (int j = 0; j < 4; ++j)   // gate: W1 slice in atoms 0, 1 and W3 slice in 2, 3
                                tma_load(b_dst + j * MN_ATOM_BYTES, gate && j >= 2 ? mp + 3 : mB,
                                         n0 + 64 * (gate ? (j & 1) : j), k0, fb);
                        }
                    }
                }
                // no copy may still be landing in shared memory when the CTA exits
                const int issued = ok ? it : it - 1;
                for (int k = issued > STAGES ? issued - STAGES : 0; k < issued; ++k)
                    mbar_wait_drain(full0 + 8 * (k % STAGES), (uint32_t)(k / STAGES) & 1u);
            }
        } else if (warp == 1) {
            if (lane == 0) {
                int it = 0, gkb = 0;   // slice and block counters over the whole run
                bool ok = true;
                for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                    const Problem& P = A.prob[problem_of(A, tile)];
                    const int nkb = (int)(s3r_cdiv(P.seg[0].K, 128) + s3r_cdiv(P.seg[1].K, 128));
                    const bool a_mn = EPI == kMixed ? P.kind == kDW : (EPI == kFwdE ? false : MN);
                    const bool b_mn = EPI == kMixed ? P.kind == kDW : (EPI == kFwdE ? true : MN);
                    const uint32_t idesc = a_mn ? idesc_f16(BM, BN, true, true)
                                                : (b_mn ? idesc_f16(BM, BN, false, true) : idesc_f16(BM, BN, false, false));
                    // one accumulator per drain unit: a 128-wide block, or kFwdUnit of them (forward)
                    const int bpu = EPI == kFwdE ? kFwdUnit : 1;
                    for (int kb = 0; kb < nkb; kb += bpu, ++gkb) {
                        const int buf = gkb & 1;
                        if (!mbar_wait(tempty0 + 8 * buf, ((uint32_t)(gkb >> 1) & 1u) ^ 1u, abrt)) {
                            ok = false;
                            break;
                        }
                        tc_after();
                        const uint32_t d_tmem = tmem + (uint32_t)(buf * BN);
                        const int kend = kb + bpu < nkb ? kb + bpu : nkb;
                        for (int b = kb; b < kend && ok; ++b) {
                            for (int h = 0; h < 2 && ok; ++h, ++it) {
                                const int s = it % STAGES;
                                if (!mbar_wait(full0 + 8 * s, (uint32_t)(it / STAGES) & 1u, abrt)) {
                                    ok = false;
                                    break;
                                }
                                tc_after();
                                const uint32_t a0 = su32(sA + s * A_STAGE), b0 = su32(sB + s * B_STAGE);
#pragma unroll
                                for (int k16 = 0; k16 < BKS / 16; ++k16) {
                                    const uint64_t ad = a_mn ? sdesc(a0 + 2048 * k16, MN_ATOM_BYTES, 1024)
                                                             : sdesc(a0 + 32 * k16, 16, 1024);
                                    const uint64_t bd = b_mn ? sdesc(b0 + 2048 * k16, MN_ATOM_BYTES, 1024)
                                                             : sdesc(b0 + 32 * k16, 16, 1024);
                                    umma_f16(d_tmem, ad, bd, idesc, (b != kb || h != 0 || k16 != 0) ? 1u : 0u);
                                }
                                umma_commit(empty0 + 8 * s);
                            }
                        }
                        if (!ok) break;
                        umma_commit(tfull0 + 8 * buf);
                    }
                }
                if (!ok) *abrt = 1;
                umma_commit(done_bar);
                mbar_wait_drain(done_bar, 0);
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
        // ------------------------------ epilogue ------------------------------
        // warp w reads TMEM lanes 32 * (w % 4) ..; two warps per lane quarter
        // split the 256 accumulator columns into halves
        const int q = warp & 3, ew = warp - EPI_WARP0, half = ew >> 2;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
        float* stage = sEpi + ew * (32 * STAGE_PITCH);
        float* cv = sCv + half * CV_FLOATS;
        const int ht = 32 * q + lane;   // thread index within the half
        int gkb = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
            const Problem& P = A.prob[problem_of(A, tile)];
            const int nkb0 = (int)s3r_cdiv(P.seg[0].K, 128), nkb1 = (int)s3r_cdiv(P.seg[1].K, 128);
            const int nkb = nkb0 + nkb1;
            int tm, tn;
            tile_coords(tile - P.tile_base, P.ntm, P.ntn, P.band_rows, tm, tn);
            const int mt = tm, nt = tn * 2 + half;   // 128-wide tile indices
            const int64_t row = (int64_t)mt * BM + 32 * q + lane;
            const bool gate = EPI == kFwdE && P.kind == kGate;
            // gate: this half owns output columns c0 .. c0 + 63, accumulators
            // 0..63 = h1 (TMEM columns 64 half ..), 64..127 = h3 (128 + 64 half ..)
            const int64_t c0 = gate ? (int64_t)tn * 128 + 64 * half : (int64_t)nt * 128;
            const uint32_t col_base = (uint32_t)(gate ? 64 * half : 128 * half);
            const uint32_t col_step = gate ? 128u - 64u : 0u;   // extra offset of chunks 4..7
            float acc[128];
            if (EPI == kFwdE) {
#pragma unroll
                for (int j = 0; j < 128; ++j) acc[j] = 0.0f;   // int32 zero
            } else if (EPI == kMixed) {
                if (P.kind != kDW) seed_tile<kDX>(P, acc, cv, row, (int64_t)mt * BM, c0, half, ht);
                else seed_tile<kDW>(P, acc, cv, row, (int64_t)mt * BM, c0, half, ht);
            } else if (EPI != kDump) {
                seed_tile<EPI>(P, acc, cv, row, (int64_t)mt * BM, c0, half, ht);
            }
            // scale of block kb, loaded one block ahead
            auto scale_of = [&](int kb) -> float {
                if (EPI == kDump) return 0.0f;
                const bool first = kb < nkb0;
                const int64_t k = first ? kb : kb - nkb0;
                const float* base = first ? P.seg[0].scale : P.seg[1].scale;
                const int64_t off = first ? mt * P.seg[0].sm + nt * P.seg[0].sn + k * P.seg[0].sk
                                          : mt * P.seg[1].sm + nt * P.seg[1].sn + k * P.seg[1].sk;
                const int64_t lim = first ? P.seg[0].nt_limit : P.seg[1].nt_limit;
                return nt < lim ? __ldg(base + off) : 0.0f;
            };
            // forward problems: one drain per kFwdUnit blocks, summed as int32 (see kFwdUnit)
            constexpr bool fwd = EPI == kFwdE;
            const int nun = fwd ? (nkb + kFwdUnit - 1) / kFwdUnit : nkb;
            float sc_next = (!fwd && nkb > 0) ? scale_of(0) : 0.0f;
            for (int kb = 0; kb < nun; ++kb, ++gkb) {
                const int buf = gkb & 1;
                const float sc = sc_next;
                if (!fwd && kb + 1 < nkb) sc_next = scale_of(kb + 1);
                // warp-uniform outcome: the tcgen05.ld below needs the whole warp
                const bool got =
                    __all_sync(0xFFFFFFFFu, mbar_wait(tfull0 + 8 * buf, (uint32_t)(gkb >> 1) & 1u, abrt));
                if (!got) {
                    ok = false;
                    *abrt = 1;
                    break;
                }
                tc_after();
                // four 16-column loads in flight per wait (64 registers next to acc[128])
#pragma unroll
                for (int c = 0; c < 8; c += 4) {
                    uint32_t r[4][16];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        tmem_ld16(lane_addr + col_base + (uint32_t)(buf * BN + 16 * (c + u)) + (c + u >= 4 ? col_step : 0u),
                                  r[u]);
                    tmem_wait_ld();
                    if (EPI == kDump) {
                        if (row < P.M) {
#pragma unroll
                            for (int u = 0; u < 4; ++u)
#pragma unroll
                                for (int j = 0; j < 16; ++j) {
                                    const int64_t col = c0 + 16 * (c + u) + j;
                                    if (col < P.N)
                                        P.dump[(row * P.N + col) * nkb + kb] =
                                            __float2int_rn(__uint_as_float(r[u][j]));
                                }
                        }
                    } else if (fwd) {
                        // exact integer partials: acc holds int32 bits
#pragma unroll
                        for (int u = 0; u < 4; ++u)
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                float& a = acc[16 * (c + u) + j];
                                a = __int_as_float(__float_as_int(a) + __float2int_rn(__uint_as_float(r[u][j])));
                            }
                    } else {
                        // acc = fma(scale, block, acc), two lanes per packed instruction
                        const float2 sc2 = make_float2(sc, sc);
#pragma unroll
                        for (int u = 0; u < 4; ++u)
#pragma unroll
                            for (int j = 0; j < 16; j += 2) {
                                const float2 a2 = f2_fma(sc2, make_float2(__uint_as_float(r[u][j]),
                                                                          __uint_as_float(r[u][j + 1])),
                                                         make_float2(acc[16 * (c + u) + j], acc[16 * (c + u) + j + 1]));
                                acc[16 * (c + u) + j] = a2.x;
                                acc[16 * (c + u) + j + 1] = a2.y;
                            }
                    }
                }
                tc_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty0 + 8 * buf);
            }
            if (EPI == kDump || !ok) continue;
            if (EPI == kFwdE) {
                if (gate) finish_gate(P, acc, row, c0);
                else finish_tile<kDX, true>(P, acc, cv, stage, row, c0, lane);
            } else if (EPI == kMixed) {
                if (P.kind != kDW) finish_tile<kDX>(P, acc, cv, stage, row, c0, lane);
                else finish_tile<kDW>(P, acc, cv, stage, row, c0, lane);
            } else {
                finish_tile<EPI>(P, acc, cv, stage, row, c0, lane);
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
    if (threadIdx.x == 0 && abort_flag) set_status(A.d_status, S3R_ERR_TIMEOUT);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (e == cudaSuccess && q == cudaDriverEntryPointSuccess && p) {
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        } else {
            (void)cudaGetLastError();
            char buf[160];
            snprintf(buf, sizeof(buf), "cudaGetDriverEntryPointByVersion: %s, query result %d", cudaGetErrorName(e),
                     (int)q);
            s3r_record_error("tensor map encoder", buf);
        }
    }
    return fn;
}

// 2-D fp16 tensor [outer, inner] (row stride row_elems), box {64, box_outer}, 128-byte swizzle, zero fill.
static int make_map(CUtensorMap* m, const void* base, int64_t inner, int64_t outer, int64_t row_elems,
                    uint32_t box_outer) {
    auto fn = encode_fn();
    if (!fn) return S3R_ERR_CUDA;
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    cuuint64_t strides[1] = {(cuuint64_t)row_elems * 2};
    cuuint32_t box[2] = {64u, box_outer};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char buf[200];
        snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled returned %d (dims %lld x %lld, box 64 x %u)", (int)r,
                 (long long)inner, (long long)outer, box_outer);
        s3r_record_error("tensor map", buf);
        return S3R_ERR_CUDA;
    }
    return S3R_OK;
}

static int sm_count() { return s3r_sm_count(); }

// Band height whose first wave of `wave` tiles touches the fewest operand
// bytes: distinct row strips x a_strip + distinct column strips x b_strip.
static int pick_band_rows(int ntm, int ntn, int wave, double a_strip, double b_strip) {
    int best = 1;
    double best_cost = -1.0;
    for (int r = 1; r <= ntm; r *= 2) {
        std::vector<char> rows(ntm, 0), cols(ntn, 0);
        int nr = 0, nc = 0;
        for (int t = 0; t < wave && t < ntm * ntn; ++t) {
            int tm, tn;
            tile_coords(t, ntm, ntn, r, tm, tn);
            if (!rows[tm]) { rows[tm] = 1; ++nr; }
            if (!cols[tn]) { cols[tn] = 1; ++nc; }
        }
        const double cost = nr * a_strip + nc * b_strip;
        if (best_cost < 0.0 || cost < best_cost) { best_cost = cost; best = r; }
    }
    return best;
}

template <int EPI, bool MN>
static int ensure_kernel() {
    static std::atomic<bool> checked{false};   // the register count is a property of the build, not the device
    const int st = s3r_kernel_smem((const void*)umma_gemm_kernel<EPI, MN>, SMEM_BYTES, "umma gemm: cudaFuncSetAttribute");
    if (st || checked.load()) return st;
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, umma_gemm_kernel<EPI, MN>);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return s3r_cuda_fail("umma gemm: cudaFuncGetAttributes", e);
    }
    if (fa.numRegs < kMinLaunchRegs || fa.numRegs > kRegsHigh) {
        char buf[160];
        snprintf(buf, sizeof(buf), "kernel built with %d registers per thread; the register split needs %d..%d",
                 fa.numRegs, kMinLaunchRegs, kRegsHigh);
        s3r_record_error("umma gemm", buf);
        return S3R_ERR_UNSUPPORTED;
    }
    checked.store(true);
    return S3R_OK;
}

// Launches the problems A.prob[0 .. A.nprob) (tile counts, bases and band
// heights filled in here); strip[i] = {bytes of one A row strip, of one B
// column strip} of problem i, for the tile order.
template <int EPI, bool MN>
static int launch(const Maps& maps, Args& A, const double (*strip)[2], cudaStream_t stream) {
    int st = ensure_kernel<EPI, MN>();
    if (st) return st;
    const int sms = sm_count();
    int64_t total = 0;
    for (int i = 0; i < A.nprob; ++i) {
        Problem& P = A.prob[i];
        const int64_t ntm = s3r_cdiv(P.M, BM), ntn = s3r_cdiv(P.N, P.kind == kGate ? BN / 2 : BN);
        if (ntm * ntn > (int64_t)1 << 30) return S3R_ERR_UNSUPPORTED;
        P.ntm = (int)ntm;
        P.ntn = (int)ntn;
        P.tile_base = (int)total;
        const int64_t tiles = ntm * ntn;
        P.band_rows = tiles ? pick_band_rows(P.ntm, P.ntn, (int)std::min<int64_t>(tiles, sms), strip[i][0],
                                             strip[i][1])
                            : 1;
        total += tiles;
        if (total > (int64_t)1 << 30) return S3R_ERR_UNSUPPORTED;
    }
    A.total_tiles = (int)total;
    if (total == 0) return S3R_OK;
    const int64_t grid = total < sms ? total : sms;   // persistent: one CTA per SM
    umma_gemm_kernel<EPI, MN><<<(unsigned)grid, THREADS, SMEM_BYTES, stream>>>(maps, A);
    S3R_CHECK_LAUNCH();
    return S3R_OK;
}

}  // namespace umma
}  // namespace s3r

using namespace s3r;

static void dx_segment(umma::Segment& g, const float* tile_scale, int64_t N, const float* eps, const int32_t* rowsum,
                       const float* v) {
    g.scale = tile_scale; g.sm = s3r_cdiv(N, kTile); g.sn = 0; g.sk = 1; g.nt_limit = INT64_MAX; g.K = N;
    g.eps = eps; g.rowsum = rowsum; g.v = v;
}

// dX problem (fp16-carried codes): A = Q [T, N], B = W [K, N] (both K-major);
// a second term (Q3, W3) contracts into the same accumulator:
// dX = Q W^T + Q3 W3^T, each term with its own tile scales and correction.
static int add_dx_problem(umma::Maps& maps, umma::Args& A, int i, const UmmaDxProblem& q, double (&strip)[2]) {
    const int64_t T = q.T, N = q.N, K = q.K, S = q.S > 0 ? q.S : q.T;
    const bool two = q.Q3 != nullptr;
    if (!s3r_aligned16(q.Q) || !s3r_aligned16(q.W) || N % 8 != 0) return S3R_ERR_ALIGN;
    if (two && (!s3r_aligned16(q.Q3) || !s3r_aligned16(q.W3))) return S3R_ERR_ALIGN;
    const int ecm = q.ec_mode == S3R_EC_DW_ONLY ? S3R_EC_NONE : q.ec_mode;   // dX is uncorrected under dW-only
    if (ecm && S < T && S % kTile != 0) {
        // the epilogue stages v for at most kNbX examples per 128-row tile
        int64_t nb = 0;
        for (int64_t m0 = 0; m0 < T; m0 += umma::BM) {
            const int64_t hi = (m0 + umma::BM - 1 < T ? m0 + umma::BM - 1 : T - 1) / S;
            if (hi - m0 / S + 1 > nb) nb = hi - m0 / S + 1;
        }
        if (nb > umma::kNbX) {
            char buf[160];
            snprintf(buf, sizeof(buf), "S = %lld lets a 128-token tile span %lld examples; the fp16-code path takes %d",
                     (long long)S, (long long)nb, umma::kNbX);
            s3r_record_error("int8_gemm_dx", buf);
            return S3R_ERR_UNSUPPORTED;
        }
    }
    CUtensorMap* m = maps.m[i];
    int st = umma::make_map(&m[0], q.Q, N, T, N, umma::BM);
    if (!st) st = umma::make_map(&m[1], q.W, N, K, N, umma::BN);
    if (!st && two) st = umma::make_map(&m[2], q.Q3, N, T, N, umma::BM);
    if (!st && two) st = umma::make_map(&m[3], q.W3, N, K, N, umma::BN);
    if (st) return st;
    if (!two) {
        m[2] = m[0];
        m[3] = m[1];
    }
    umma::Problem& P = A.prob[i];
    P = umma::Problem{};
    P.M = T; P.N = K; P.kind = umma::kDX;
    dx_segment(P.seg[0], q.tile_scale, N, q.eps, q.rowsum, q.v);
    if (two) dx_segment(P.seg[1], q.tile_scale3, N, q.eps3, q.rowsum3, q.v3);
    P.C = q.dX; P.ldc = K; P.dump = q.dump; P.s_row = q.s_x; P.ec_mode = ecm; P.S = S;
    P.accumulate = q.accumulate;
    // bytes per row strip of A (BM rows of Q over the contraction) and per column strip of B (BN rows of W)
    const double kbytes = 2.0 * (double)N * (two ? 2 : 1);
    strip[0] = umma::BM * kbytes;
    strip[1] = umma::BN * kbytes;
    return S3R_OK;
}

// dW problem (fp16-carried codes): A = X [T, K], B = Q [T, N] (both MN-major, contracted over T).
static int add_dw_problem(umma::Maps& maps, umma::Args& A, int i, const UmmaDwProblem& q, double (&strip)[2]) {
    const int64_t T = q.T, K = q.K, N = q.N, S = q.S > 0 ? q.S : q.T;
    if (!s3r_aligned16(q.Q) || !s3r_aligned16(q.X) || N % 8 != 0 || K % 8 != 0) return S3R_ERR_ALIGN;
    CUtensorMap* m = maps.m[i];
    int st = umma::make_map(&m[0], q.X, K, T, K, 64);
    if (!st) st = umma::make_map(&m[1], q.Q, N, T, N, 64);
    if (st) return st;
    m[2] = m[0];
    m[3] = m[1];
    umma::Problem& P = A.prob[i];
    P = umma::Problem{};
    P.M = K; P.N = N; P.kind = umma::kDW;
    umma::Segment& g = P.seg[0];
    g.scale = q.tile_scale; g.sm = 0; g.sn = 1; g.sk = s3r_cdiv(N, kTile); g.nt_limit = s3r_cdiv(N, kTile);
    g.K = T;
    P.C = q.dW; P.ldc = N; P.dump = q.dump; P.s_col = q.s_w; P.S = S;
    P.ec_mode = q.ec_mode == S3R_EC_DW_ONLY ? S3R_EC_TWO_WAY : q.ec_mode;   // dW carries the whole correction
    P.B = q.S > 0 ? T / q.S : 1; P.colmean = q.colmean; P.mu = q.mu; P.xsum = q.xsum; P.p = q.p;
    const double kbytes = 2.0 * (double)T;   // per output row / column over the contraction
    strip[0] = umma::BM * kbytes;
    strip[1] = umma::BN * kbytes;
    return S3R_OK;
}

// Forward problems (fp16-carried codes): A = X [T, K] K-major, B = W [K, N]
// MN-major (as stored), unit block scales.  kFwd writes Y [T, N] fp32 =
// (acc * s_x[t]) * s_w[n]; kGate contracts X with W1 and W3 at once and writes
// h1, h3 and a (bf16 [T, N], row stride N) through the SwiGLU gate.
static int add_fwd_problem(umma::Maps& maps, umma::Args& A, int i, const void* X, const float* s_x, const void* W,
                           const float* s_w, const void* W3, const float* s_w3, int64_t T, int64_t K, int64_t N,
                           float* Y, uint16_t* const* gate_out, double (&strip)[2]) {
    const bool gate = W3 != nullptr;
    if (!s3r_aligned16(X) || !s3r_aligned16(W) || K % 8 != 0 || N % 8 != 0) return S3R_ERR_ALIGN;
    if (gate && !s3r_aligned16(W3)) return S3R_ERR_ALIGN;
    CUtensorMap* m = maps.m[i];
    int st = umma::make_map(&m[0], X, K, T, K, umma::BM);
    if (!st) st = umma::make_map(&m[1], W, N, K, N, 64);
    if (!st && gate) st = umma::make_map(&m[3], W3, N, K, N, 64);
    if (st) return st;
    m[2] = m[0];
    if (!gate) m[3] = m[1];
    umma::Problem& P = A.prob[i];
    P = umma::Problem{};
    P.M = T; P.N = N; P.kind = gate ? umma::kGate : umma::kFwd;
    umma::Segment& g = P.seg[0];
    g.scale = nullptr; g.sm = g.sn = g.sk = 0; g.nt_limit = INT64_MAX; g.K = K;
    P.f_row = s_x; P.f_col = s_w; P.f_col3 = s_w3;
    P.C = Y; P.ldc = N; P.S = T;
    if (gate)
        for (int j = 0; j < 3; ++j) P.gate_out[j] = gate_out[j];
    strip[0] = umma::BM * 2.0 * (double)K;
    strip[1] = umma::BN * 2.0 * (double)K;
    return S3R_OK;
}

int umma_fwd(const void* X, const float* s_x, const void* W, const float* s_w, const void* W3, const float* s_w3,
             int64_t T, int64_t K, int64_t N, float* Y, uint16_t* h1, uint16_t* h3, uint16_t* a, int* d_status,
             cudaStream_t stream) {
    thread_local umma::Maps maps;
    thread_local umma::Args A;
    std::memset(&A, 0, sizeof(A));
    double strip[1][2];
    uint16_t* outs[3] = {h1, h3, a};
    const int st = add_fwd_problem(maps, A, 0, X, s_x, W, s_w, W3, s_w3, T, K, N, Y, outs, strip[0]);
    if (st) return st;
    A.nprob = 1;
    A.d_status = d_status;
    return umma::launch<umma::kFwdE, false>(maps, A, strip, stream);
}

int umma_dx_group(const UmmaDxProblem* probs, int n, int* d_status, cudaStream_t stream) {
    if (n < 1 || n > umma::kMaxProb) return S3R_ERR_ARG;
    thread_local umma::Maps maps;   // host staging of the launch's parameters (copied at launch)
    thread_local umma::Args A;
    std::memset(&A, 0, sizeof(A));
    double strip[umma::kMaxProb][2];
    bool dump = false;
    for (int i = 0; i < n; ++i) {
        const int st = add_dx_problem(maps, A, i, probs[i], strip[i]);
        if (st) return st;
        dump = dump || probs[i].dump;
    }
    A.nprob = n;
    A.d_status = d_status;
    if (dump) return umma::launch<umma::kDump, false>(maps, A, strip, stream);
    return umma::launch<umma::kDX, false>(maps, A, strip, stream);
}

int umma_dw_group(const UmmaDwProblem* probs, int n, int* d_status, cudaStream_t stream) {
    if (n < 1 || n > umma::kMaxProb) return S3R_ERR_ARG;
    thread_local umma::Maps maps;
    thread_local umma::Args A;
    std::memset(&A, 0, sizeof(A));
    double strip[umma::kMaxProb][2];
    bool dump = false;
    for (int i = 0; i < n; ++i) {
        const int st = add_dw_problem(maps, A, i, probs[i], strip[i]);
        if (st) return st;
        dump = dump || probs[i].dump;
    }
    A.nprob = n;
    A.d_status = d_status;
    if (dump) return umma::launch<umma::kDump, true>(maps, A, strip, stream);
    return umma::launch<umma::kDW, true>(maps, A, strip, stream);
}

// dX and dW problems in one launch (no dumps).  Problems run in the order of
// their per-tile contraction length, longest first, so the short tiles at the
// end of the round-robin fill in behind the long ones.
int umma_mixed_group(const UmmaDxProblem* dx, int ndx, const UmmaDwProblem* dw, int ndw, int* d_status,
                     cudaStream_t stream) {
    const int n = ndx + ndw;
    if (ndx < 0 || ndw < 0 || n < 1 || n > umma::kMaxProb) return S3R_ERR_ARG;
    thread_local umma::Maps maps;
    thread_local umma::Args A;
    std::memset(&A, 0, sizeof(A));
    double strip[umma::kMaxProb][2];
    // order: per-tile 128-blocks descending (stable)
    int order[umma::kMaxProb];
    int64_t blocks[umma::kMaxProb];
    for (int i = 0; i < n; ++i) {
        order[i] = i;
        blocks[i] = i < ndx ? s3r_cdiv(dx[i].N, 128) * (dx[i].Q3 ? 2 : 1) : s3r_cdiv(dw[i - ndx].T, 128);
    }
    std::stable_sort(order, order + n, [&](int a, int b) { return blocks[a] > blocks[b]; });
    for (int k = 0; k < n; ++k) {
        const int i = order[k];
        if (i < ndx && dx[i].dump) return S3R_ERR_ARG;
        if (i >= ndx && dw[i - ndx].dump) return S3R_ERR_ARG;
        const int st = i < ndx ? add_dx_problem(maps, A, k, dx[i], strip[k])
                               : add_dw_problem(maps, A, k, dw[i - ndx], strip[k]);
        if (st) return st;
    }
    A.nprob = n;
    A.d_status = d_status;
    return umma::launch<umma::kMixed, false>(maps, A, strip, stream);
}

int umma_gemm_dx2(const void* Q, const float* tile_scale, const void* W, const float* eps, const int32_t* rowsum,
                  const float* v, const void* Q3, const float* tile_scale3, const void* W3, const float* eps3,
                  const int32_t* rowsum3, const float* v3, int64_t T, int64_t N, int64_t K, const float* s_x,
                  int ec_mode, int64_t S, float* dX, int accumulate, int32_t* dump, int* d_status,
                  cudaStream_t stream) {
    const UmmaDxProblem q{Q, tile_scale, W, eps, rowsum, v, Q3, tile_scale3, W3, eps3, rowsum3, v3,
                          T, N, K, s_x, ec_mode, S, dX, accumulate, dump};
    return umma_dx_group(&q, 1, d_status, stream);
}

int umma_gemm_dx(const void* Q, const float* tile_scale, const void* W, int64_t T, int64_t N, int64_t K,
                 const float* s_x, int ec_mode, const float* eps, const int32_t* rowsum, const float* v, int64_t S,
                 float* dX, int accumulate, int32_t* dump, int* d_status, cudaStream_t stream) {
    return umma_gemm_dx2(Q, tile_scale, W, eps, rowsum, v, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, T, N,
                         K, s_x, ec_mode, S, dX, accumulate, dump, d_status, stream);
}

int umma_gemm_dw(const void* X, const void* Q, const float* tile_scale, int64_t T, int64_t K, int64_t N,
                 const float* s_w, int ec_mode, const float* colmean, const float* mu, const int32_t* xsum,
                 const float* p, int64_t S, float* dW, int32_t* dump, int* d_status, cudaStream_t stream) {
    const UmmaDwProblem q{X, Q, tile_scale, T, K, N, s_w, ec_mode, colmean, mu, xsum, p, S, dW, dump};
    return umma_dw_group(&q, 1, d_status, stream);
}

// ---------------------------------------------------------------------------
// C ABI of the forward GEMMs
// ---------------------------------------------------------------------------
static int fwd_args(const void* X8, const float* s_x, const void* W8, const float* s_w, int code_format, int64_t T,
                    int64_t K, int64_t N) {
    if (T < 0 || K < 0 || N < 0) return S3R_ERR_ARG;
    if (code_format != S3R_CODES_S8 && code_format != S3R_CODES_F16) return S3R_ERR_ARG;
    if (code_format != S3R_CODES_F16) {
        s3r_record_error("int8_gemm_fwd", "the forward runs on fp16-carried codes (S3R_CODES_F16) only");
        return S3R_ERR_UNSUPPORTED;
    }
    if (T > 0 && N > 0 && K > 0 && (!X8 || !s_x || !W8 || !s_w)) return S3R_ERR_ARG;
    return S3R_OK;
}

extern "C" int int8_gemm_fwd(const void* X8, const float* s_x, const void* W8, const float* s_w, int code_format,
                             int64_t T, int64_t K, int64_t N, float* Y, int* d_status, cudaStream_t stream) {
    int st = fwd_args(X8, s_x, W8, s_w, code_format, T, K, N);
    if (st) return st;
    if (T == 0 || N == 0) return S3R_OK;
    if (!Y) return S3R_ERR_ARG;
    if (K == 0) {
        const cudaError_t e = cudaMemsetAsync(Y, 0, (size_t)(T * N) * sizeof(float), stream);
        return e == cudaSuccess ? S3R_OK : s3r_cuda_fail("int8_gemm_fwd: cudaMemsetAsync", e);
    }
    return umma_fwd(X8, s_x, W8, s_w, nullptr, nullptr, T, K, N, Y, nullptr, nullptr, nullptr, d_status, stream);
}

extern "C" int int8_gemm_fwd_swiglu(const void* X8, const float* s_x, const void* W1_8, const float* s_w1,
                                    const void* W3_8, const float* s_w3, int code_format, int64_t T, int64_t K,
                                    int64_t F, void* h1, void* h3, void* a, int* d_status, cudaStream_t stream) {
    int st = fwd_args(X8, s_x, W1_8, s_w1, code_format, T, K, F);
    if (st) return st;
    if (T == 0 || F == 0) return S3R_OK;
    if (!h1 || !h3 || (K > 0 && (!W3_8 || !s_w3))) return S3R_ERR_ARG;
    if (K == 0) {   // h1 = h3 = 0, a = silu(0) * 0 = 0
        for (void* p : {h1, h3, a}) {
            if (!p) continue;
            const cudaError_t e = cudaMemsetAsync(p, 0, (size_t)(T * F) * 2, stream);
            if (e != cudaSuccess) return s3r_cuda_fail("int8_gemm_fwd_swiglu: cudaMemsetAsync", e);
        }
        return S3R_OK;
    }
    return umma_fwd(X8, s_x, W1_8, s_w1, W3_8, s_w3, T, K, F, nullptr, static_cast<uint16_t*>(h1),
                    static_cast<uint16_t*>(h3), static_cast<uint16_t*>(a), d_status, stream);
}
