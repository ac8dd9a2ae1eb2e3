// gemm_umma.cu -- the INT8 backward GEMMs on the 5th-generation tensor cores
// (tcgen05, sm_103a), with the codes carried exactly in fp16.
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

#include <cuda.h>
#include <cudaTypedefs.h>
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

enum Epi { kDX = 0, kDW = 1, kDump = 2 };

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

struct Args {
    int64_t M, N;                // C[M, N] = sum over segments of sum_k A[m, k] B[n, k]
    Segment seg[2];              // seg[1].K == 0 when there is one segment
    float* C;
    int64_t ldc;
    int32_t* dump;
    const float* s_row;          // dX: 1/s_x[row] rescale
    const float* s_col;          // dW: 1/s_w[col] rescale
    int ec_mode;
    int64_t S, B;
    const float* colmean;
    const float* mu;
    const int32_t* xsum;
    const float* p;
    int accumulate;
    int* d_status;
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
__device__ __forceinline__ void seed_tile(const Args& P, float (&acc)[128], float* cv, int64_t row, int64_t m0,
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
            for (int i = 0; i < kNbX; ++i)
                cv[256 + (g * kNbX + i) * 128 + ht] =
                    (on && cin && b_lo + i <= b_hi) ? __ldg(P.seg[g].v + (b_lo + i) * P.N + cc) : 0.0f;
        }
        half_bar(half);
        const float ep0 = in ? __ldg(P.seg[0].eps + row) : 0.0f;
        const float ep1 = (in && P.seg[1].K > 0) ? __ldg(P.seg[1].eps + row) : 0.0f;
        const int i_row = in ? (int)(row / P.S - b_lo) : 0;
        const float* rs0 = cv;
        const float* v0 = cv + 256 + i_row * 128;
#pragma unroll
        for (int j4 = 0; j4 < 128; j4 += 4) {
            const float4 r = lds4(rs0 + j4), w = lds4(v0 + j4);
            acc[j4 + 0] = -fmaf(ep0, r.x, w.x);
            acc[j4 + 1] = -fmaf(ep0, r.y, w.y);
            acc[j4 + 2] = -fmaf(ep0, r.z, w.z);
            acc[j4 + 3] = -fmaf(ep0, r.w, w.w);
        }
        if (P.seg[1].K > 0) {
            const float* rs1 = cv + 128;
            const float* v1 = cv + 256 + (kNbX + i_row) * 128;
#pragma unroll
            for (int j4 = 0; j4 < 128; j4 += 4) {
                const float4 r = lds4(rs1 + j4), w = lds4(v1 + j4);
                acc[j4 + 0] = acc[j4 + 0] - fmaf(ep1, r.x, w.x);
                acc[j4 + 1] = acc[j4 + 1] - fmaf(ep1, r.y, w.y);
                acc[j4 + 2] = acc[j4 + 2] - fmaf(ep1, r.z, w.z);
                acc[j4 + 3] = acc[j4 + 3] - fmaf(ep1, r.w, w.w);
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
#pragma unroll
                for (int j4 = 0; j4 < 128; j4 += 4) {
                    const float4 c4 = lds4(cm + j4);
                    acc[j4 + 0] = fmaf(xs, c4.x, acc[j4 + 0]);
                    acc[j4 + 1] = fmaf(xs, c4.y, acc[j4 + 1]);
                    acc[j4 + 2] = fmaf(xs, c4.z, acc[j4 + 2]);
                    acc[j4 + 3] = fmaf(xs, c4.w, acc[j4 + 3]);
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
template <int EPI>
__device__ __forceinline__ void finish_tile(const Args& P, float (&acc)[128], const float* cv, float* stage,
                                            int64_t row, int64_t c0, int lane) {
    if (EPI == kDX && P.s_row) {
        const float rinv = row < P.M ? __frcp_rn(__ldg(P.s_row + row)) : 1.0f;
#pragma unroll
        for (int j = 0; j < 128; ++j) acc[j] = acc[j] * rinv;
    }
    if (EPI == kDW && P.s_col) {
#pragma unroll
        for (int j4 = 0; j4 < 128; j4 += 4) {
            const float4 r = lds4(cv + j4);
            acc[j4 + 0] *= r.x;
            acc[j4 + 1] *= r.y;
            acc[j4 + 2] *= r.z;
            acc[j4 + 3] *= r.w;
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

// 12 warps: one SM sub-partition hosts three of them, one per warpgroup, so the
// launch is capped at 168 registers per thread; after the split a
// sub-partition holds (40 + 216 + 216) * 32 = 15104 of its 16384.
template <int EPI, bool MN>
__global__ void __launch_bounds__(THREADS, 1)
    umma_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmB0,
                     const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1, Args P) {
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
    const int nkb0 = (int)s3r_cdiv(P.seg[0].K, 128), nkb1 = (int)s3r_cdiv(P.seg[1].K, 128);
    const int nkb = nkb0 + nkb1;                 // 128-wide blocks per tile
    // tile counts fit 32 bits: the host caps M and N far below 2^31 * 128
    const int ntn = (int)s3r_cdiv(P.N, BN), ntiles = (int)s3r_cdiv(P.M, BM) * ntn;

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
                asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmA0) : "memory");
                asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmB0) : "memory");
                if (nkb1) {
                    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmA1) : "memory");
                    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmB1) : "memory");
                }
                int it = 0;   // slice counter over the whole persistent run
                bool ok = true;
                for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                    const int32_t m0 = (tile / ntn) * BM, n0 = (tile % ntn) * BN;
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
                        const CUtensorMap* mA = second ? &tmA1 : &tmA0;
                        const CUtensorMap* mB = second ? &tmB1 : &tmB0;
                        const int32_t k0 = (second ? sl - 2 * nkb0 : sl) * BKS;
                        const uint32_t a_dst = su32(sA + s * A_STAGE), b_dst = su32(sB + s * B_STAGE);
                        if (!MN) {
                            tma_load(a_dst, mA, k0, m0, fb);
                            tma_load(b_dst, mB, k0, n0, fb);
                        } else {
                            tma_load(a_dst, mA, m0, k0, fb);
                            tma_load(a_dst + MN_ATOM_BYTES, mA, m0 + 64, k0, fb);
#pragma unroll
                            for (int j = 0; j < 4; ++j) tma_load(b_dst + j * MN_ATOM_BYTES, mB, n0 + 64 * j, k0, fb);
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
                constexpr uint32_t idesc = idesc_f16(BM, BN, MN, MN);
                int it = 0, gkb = 0;   // slice and block counters over the whole run
                bool ok = true;
                for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                    for (int kb = 0; kb < nkb; ++kb, ++gkb) {
                        const int buf = gkb & 1;
                        if (!mbar_wait(tempty0 + 8 * buf, ((uint32_t)(gkb >> 1) & 1u) ^ 1u, abrt)) {
                            ok = false;
                            break;
                        }
                        tc_after();
                        const uint32_t d_tmem = tmem + (uint32_t)(buf * BN);
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
                                uint64_t ad, bd;
                                if (!MN) {
                                    ad = sdesc(a0 + 32 * k16, 16, 1024);
                                    bd = sdesc(b0 + 32 * k16, 16, 1024);
                                } else {
                                    ad = sdesc(a0 + 2048 * k16, MN_ATOM_BYTES, 1024);
                                    bd = sdesc(b0 + 2048 * k16, MN_ATOM_BYTES, 1024);
                                }
                                umma_f16(d_tmem, ad, bd, idesc, (h | k16) != 0);
                            }
                            umma_commit(empty0 + 8 * s);
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
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(128 * half);
        float* stage = sEpi + ew * (32 * STAGE_PITCH);
        float* cv = sCv + half * CV_FLOATS;
        const int ht = 32 * q + lane;   // thread index within the half
        int gkb = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
            const int mt = tile / ntn, nt = (tile % ntn) * 2 + half;   // 128-wide tile indices
            const int64_t row = (int64_t)mt * BM + 32 * q + lane;
            const int64_t c0 = (int64_t)nt * 128;
            float acc[128];
            if (EPI != kDump) seed_tile<EPI>(P, acc, cv, row, (int64_t)mt * BM, c0, half, ht);
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
            float sc_next = nkb > 0 ? scale_of(0) : 0.0f;
            for (int kb = 0; kb < nkb; ++kb, ++gkb) {
                const int buf = gkb & 1;
                const float sc = sc_next;
                if (kb + 1 < nkb) sc_next = scale_of(kb + 1);
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
                    for (int u = 0; u < 4; ++u) tmem_ld16(lane_addr + (uint32_t)(buf * BN + 16 * (c + u)), r[u]);
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
                    } else {
#pragma unroll
                        for (int u = 0; u < 4; ++u)
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                acc[16 * (c + u) + j] = fmaf(sc, __uint_as_float(r[u][j]), acc[16 * (c + u) + j]);
                    }
                }
                tc_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty0 + 8 * buf);
            }
            if (EPI == kDump || !ok) continue;
            finish_tile<EPI>(P, acc, cv, stage, row, c0, lane);
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
    if (threadIdx.x == 0 && abort_flag) set_status(P.d_status, S3R_ERR_TIMEOUT);
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

static int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 148;
    }
    return n;
}

template <int EPI, bool MN>
static int launch(const CUtensorMap& a0, const CUtensorMap& b0, const CUtensorMap& a1, const CUtensorMap& b1,
                  const Args& P, cudaStream_t stream) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e =
            cudaFuncSetAttribute(umma_gemm_kernel<EPI, MN>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return s3r_cuda_fail("umma gemm: cudaFuncSetAttribute", e);
        }
        cudaFuncAttributes fa{};
        e = cudaFuncGetAttributes(&fa, umma_gemm_kernel<EPI, MN>);
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
        attr = true;
    }
    const int64_t ntiles = s3r_cdiv(P.M, BM) * s3r_cdiv(P.N, BN);
    if (ntiles == 0) return S3R_OK;
    const int64_t grid = ntiles < sm_count() ? ntiles : sm_count();   // persistent: one CTA per SM
    umma_gemm_kernel<EPI, MN><<<(unsigned)grid, THREADS, SMEM_BYTES, stream>>>(a0, b0, a1, b1, P);
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

// dX [T, K] from fp16-carried codes: A = Q [T, N], B = W [K, N] (both K-major);
// with a second term (Q3, W3) the kernel contracts both into one accumulator:
// dX = Q W^T + Q3 W3^T, each term with its own tile scales and correction.
int umma_gemm_dx2(const void* Q, const float* tile_scale, const void* W, const float* eps, const int32_t* rowsum,
                  const float* v, const void* Q3, const float* tile_scale3, const void* W3, const float* eps3,
                  const int32_t* rowsum3, const float* v3, int64_t T, int64_t N, int64_t K, const float* s_x,
                  int ec_mode, int64_t S, float* dX, int accumulate, int32_t* dump, int* d_status,
                  cudaStream_t stream) {
    if (!s3r_aligned16(Q) || !s3r_aligned16(W) || N % 8 != 0) return S3R_ERR_ALIGN;
    if (Q3 && (!s3r_aligned16(Q3) || !s3r_aligned16(W3))) return S3R_ERR_ALIGN;
    CUtensorMap ma, mb, ma3, mb3;
    int st = umma::make_map(&ma, Q, N, T, N, umma::BM);
    if (!st) st = umma::make_map(&mb, W, N, K, N, umma::BN);
    if (!st && Q3) st = umma::make_map(&ma3, Q3, N, T, N, umma::BM);
    if (!st && Q3) st = umma::make_map(&mb3, W3, N, K, N, umma::BN);
    if (st) return st;
    if (!Q3) {
        ma3 = ma;
        mb3 = mb;
    }
    if (ec_mode && S > 0 && S < T && S % kTile != 0) {
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
    umma::Args P{};
    P.M = T; P.N = K;
    dx_segment(P.seg[0], tile_scale, N, eps, rowsum, v);
    if (Q3) dx_segment(P.seg[1], tile_scale3, N, eps3, rowsum3, v3);
    P.C = dX; P.ldc = K; P.dump = dump; P.s_row = s_x; P.ec_mode = ec_mode; P.S = S > 0 ? S : T;
    P.accumulate = accumulate; P.d_status = d_status;
    if (dump) return umma::launch<umma::kDump, false>(ma, mb, ma3, mb3, P, stream);
    return umma::launch<umma::kDX, false>(ma, mb, ma3, mb3, P, stream);
}

int umma_gemm_dx(const void* Q, const float* tile_scale, const void* W, int64_t T, int64_t N, int64_t K,
                 const float* s_x, int ec_mode, const float* eps, const int32_t* rowsum, const float* v, int64_t S,
                 float* dX, int accumulate, int32_t* dump, int* d_status, cudaStream_t stream) {
    return umma_gemm_dx2(Q, tile_scale, W, eps, rowsum, v, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, T, N,
                         K, s_x, ec_mode, S, dX, accumulate, dump, d_status, stream);
}

// dW [K, N] from fp16-carried codes: A = X [T, K], B = Q [T, N] (both MN-major, contracted over T).
int umma_gemm_dw(const void* X, const void* Q, const float* tile_scale, int64_t T, int64_t K, int64_t N,
                 const float* s_w, int ec_mode, const float* colmean, const float* mu, const int32_t* xsum,
                 const float* p, int64_t S, float* dW, int32_t* dump, int* d_status, cudaStream_t stream) {
    if (!s3r_aligned16(Q) || !s3r_aligned16(X) || N % 8 != 0 || K % 8 != 0) return S3R_ERR_ALIGN;
    CUtensorMap ma, mb;
    int st = umma::make_map(&ma, X, K, T, K, 64);
    if (st) return st;
    st = umma::make_map(&mb, Q, N, T, N, 64);
    if (st) return st;
    umma::Args P{};
    P.M = K; P.N = N;
    umma::Segment& g = P.seg[0];
    g.scale = tile_scale; g.sm = 0; g.sn = 1; g.sk = s3r_cdiv(N, kTile); g.nt_limit = s3r_cdiv(N, kTile); g.K = T;
    P.C = dW; P.ldc = N; P.dump = dump; P.s_col = s_w; P.ec_mode = ec_mode; P.S = S > 0 ? S : T;
    P.B = S > 0 ? T / S : 1; P.colmean = colmean; P.mu = mu; P.xsum = xsum; P.p = p; P.d_status = d_status;
    if (dump) return umma::launch<umma::kDump, true>(ma, mb, ma, mb, P, stream);
    return umma::launch<umma::kDW, true>(ma, mb, ma, mb, P, stream);
}
