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
//   warps 2, 3  helpers: copy each tile's epilogue vectors (rescale factors,
//               correction terms) into a shared-memory side buffer with
//               cp.async while the tile's first blocks run;
//   warps 4..11 epilogue: per 128-K block, tcgen05.ld their 32 TMEM lanes x
//               128 columns, acc = fma(scale, block, acc) in registers; after
//               block kCorrBlock they subtract the correction (from the side
//               buffer), at the end of the tile rescale by 1/s and hand the
//               tile to the TMA engine (bulk tensor stores from small
//               swizzled staging buffers), while the producer and the MMA
//               issuer already run the next tile.
// Warpgroup 0 gives registers to the epilogue warpgroups (setmaxnreg), so a
// drain keeps four TMEM loads in flight next to the 128 accumulators.
// The tile boundary is what the two TMEM accumulators must hide (about two
// blocks of MMA time), so nothing on it waits for global memory: the side
// data is already in shared memory and the stores are asynchronous.
// The activation gradient may contract two operand pairs into one
// accumulator (dX = Q1 W1^T + Q3 W3^T), each with its own scales.
// A third instantiation (kMixedG) can end one dX problem -- the activation
// gradient dA of the SwiGLU block's down projection -- with the SwiGLU glue
// and the quantization of dh1 and dh3 instead of a store (glue_tile below).
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
#include "deal_plan.h"

namespace s3r {
namespace umma {

constexpr int BM = 128, BN = 256, BKS = 64, STAGES = 4;
constexpr int A_STAGE = BM * BKS * 2;       // 16 KiB
constexpr int B_STAGE = BN * BKS * 2;       // 32 KiB
constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
constexpr int MN_ATOM_BYTES = BKS * 128;    // one 64-wide MN atom column over a 64-deep K slice: 8 KiB
constexpr int THREADS = 384;               // three warpgroups
constexpr int EPI_WARP0 = 4;                // epilogue warps 4..11 (warpgroups 1 and 2)
// Register split (setmaxnreg): warpgroup 0 (producer, MMA issuer, two
// helpers) drops to kRegsLow, the epilogue warpgroups rise to kRegsHigh.  The
// launch holds regs_per_thread * 384 registers; the split needs
// kRegsLow * 128 + kRegsHigh * 256 of them, so the host refuses to launch a
// build whose per-thread count is below kMinLaunchRegs (an increase that the
// pool cannot satisfy would wait forever).
constexpr int kRegsLow = 56, kRegsHigh = 216;
// The glue instantiation gives warpgroup 0 the whole remainder of a
// 168-register launch (its helpers also bring the glue's side data in).
constexpr int kRegsLowGlue = 72;
constexpr int kMinLaunchRegs = (kRegsLowGlue * 128 + kRegsHigh * 256 + 383) / 384;
static_assert(kRegsLow <= kRegsLowGlue, "the launch check covers both splits");
constexpr int EPI_WARPS = 8;
// Output staging of the TMA stores: per epilogue warp two buffers of 32 rows x
// 8 fp32 columns (1 KiB each, 32-byte swizzle), so the warp fills one while
// the TMA engine still reads the other.
constexpr int OUT_COLS = 8;
constexpr int OUT_BUF_BYTES = 32 * OUT_COLS * 4;
constexpr int OUT_STAGE_BYTES = EPI_WARPS * 2 * OUT_BUF_BYTES;   // 16 KiB
constexpr int kNbX = 4;                     // dX: examples one 128-row tile may span (S >= 43)
constexpr int kBch = 8;                     // dW: examples whose correction vectors are staged per round
// Side data of one tile, copied into shared memory by the two helper warps
// while the tile's first blocks run (offsets in floats; rows of the tile are
// its 128 output rows, columns its 256 output columns):
//   dX: 1/s_x[row] | eps_g[row] (g < 2) | rowsum_g[col] | v_g[b_lo + i][col] (i < kNbX)
//   dW: 1/s_w[col] | p[row] | xsum[b][row] | colmean[b][col] - mu[b] for a round
//       of kBch examples (B > kBch takes several rounds, each refilling the
//       last two arrays)
constexpr int SX_ROWSC = 0, SX_EPS = 128, SX_RS = SX_EPS + 2 * 128, SX_V = SX_RS + 2 * 256;
constexpr int SX_END = SX_V + 2 * kNbX * 256;
constexpr int SW_COLSC = 0, SW_P = 256, SW_XS = SW_P + 128, SW_CM = SW_XS + kBch * 128;
constexpr int SW_END = SW_CM + kBch * 256;
constexpr int SIDE_FLOATS = SX_END > SW_END ? SX_END : SW_END;
// The glue problem has one contraction term, so the second term's v slab holds
// the glue's side data instead: s_x[row] (the fold, not its reciprocal) and
// s_w1, s_w3 of the tile's 256 columns.
constexpr int SG_SX = SX_V + kNbX * 256, SG_SW1 = SG_SX + 128, SG_SW3 = SG_SW1 + 256, SG_END = SG_SW3 + 256;
static_assert(SG_END <= SX_END, "glue side data inside the dX side layout");
// The correction enters the accumulators after block kCorrBlock of a tile,
// which leaves the helpers a few blocks to bring the tile's side data in.
constexpr int kCorrBlock = 3;
constexpr uint32_t TMEM_COLS = 512;
// + three exchange barriers per epilogue warpgroup for the glue epilogue
constexpr int NUM_BARS = 2 * STAGES + 7 + 6;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + OUT_STAGE_BYTES + SIDE_FLOATS * 4 + 1024 + NUM_BARS * 8 + 16;
static_assert(SMEM_BYTES + 64 <= 232448, "shared memory budget of one sm_103a CTA");
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait

// Epilogue kinds; a kMixed launch takes each problem's kind (kDX or kDW) from
// the problem, a kFwdE launch (forward problems only) too (kFwd or kGate).
// The forward gets its own instantiation so that the backward kernels carry
// none of its code.
enum Epi { kDX = 0, kDW = 1, kDump = 2, kMixed = 3, kFwdE = 4, kMixedG = 6 };
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
    int accumulate;              // C += result (an add-reduction store)
    int c_tma;                   // C is addressable by the TMA engine (map 4 of the problem)
};

// A launch: up to kMaxProb problems (of one kind, or mixed), their tiles numbered one
// after another; each problem has up to five tensor maps (A and B of each
// segment, and the output C).  Both live in the constant parameter space (__grid_constant__),
// so indexing them with a run-time problem number costs no copy.
constexpr int kMaxProb = 24;
// The SwiGLU glue of a kMixedG launch (see UmmaGlue): problem `prob` stores
// no dA; its epilogue writes the codes of dh1 and dh3 instead.
struct Glue {
    int prob;                    // launch problem carrying the glue (-1: none)
    int rtne;                    // 1: round to nearest even; 0: SR with one threshold per row
    int thr;                     // row thresholds: 0 per token, 1 per token (7-bit), 2 per example
    uint32_t seed_lo, tid1, tid3;
    int64_t S;                   // tokens per example (thr == 2)
    const uint16_t* h1;
    const uint16_t* h3;
    int64_t ldh;
    const float* s_x;
    const float* s_w1;
    const float* s_w3;
    uint16_t* Q1;
    uint16_t* Q3;
    float* scale1;
    float* scale3;
    float* tok1;
    float* tok3;
    float* col1;
    float* col3;
    int64_t ntc;                 // 128-wide column tiles of dh1 (ceil(F / 128))
};
struct Args {
    Problem prob[kMaxProb];
    int nprob;
    int total_tiles;
    int* d_status;
    Glue glue;
    // How problem i's tiles are dealt to the CTAs of a mixed launch (next_tile):
    // first deal_m[i] rounds over the deal_w[i] CTAs deal_s[i], deal_s[i] + 1, ...
    // (cyclic), then round robin over all CTAs from deal_s[i].
    int deal_s[kMaxProb], deal_w[kMaxProb], deal_m[kMaxProb];
};
struct Maps {
    CUtensorMap m[kMaxProb][5];
};
static_assert(sizeof(Maps) + sizeof(Args) <= 32764, "kernel parameters beyond the 32764-byte limit");

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
// limit_ns or as soon as another role raised the abort flag.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t limit_ns = kWaitNs) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = gtime();
    while (!mbar_try(bar, parity)) {
        if (*abort_flag) return false;
        if (gtime() - t0 > limit_ns) return false;
    }
    return true;
}

// Test hook: mbar_wait on a barrier that nothing arrives on, with a short
// limit; with raise_abort a second warp raises the abort flag after about a
// millisecond instead.  The waiter records how long it waited and, having
// given up, sets S3R_ERR_TIMEOUT as the kernels do.
__global__ void __launch_bounds__(64) wait_probe_kernel(uint64_t limit_ns, int raise_abort, int* d_status,
                                                        unsigned long long* waited_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_s;
    const uint32_t b = su32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 32 && raise_abort) {
        const uint64_t t0 = gtime();
        while (gtime() - t0 < 1000000ull) {}
        *reinterpret_cast<volatile int*>(&abort_s) = 1;
    } else if (threadIdx.x == 0) {
        const uint64_t t0 = gtime();
        const bool ok = mbar_wait(b, 0u, &abort_s, limit_ns);
        *waited_ns = gtime() - t0;
        if (!ok) set_status(d_status, S3R_ERR_TIMEOUT);
    }
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
// thread i writes 16 consecutive 32-bit columns of lane (base + i)
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float4 lds4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// ---------------------------------------------------------------------------
// Side data.  The two helper warps (64 threads) copy a tile's epilogue vectors
// from global memory into the side buffer with cp.async (no registers held,
// zero fill past the tensor ends), then convert them in place: reciprocals of
// the rescale factors, int32 sums to float, colmean - mu.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(float* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(su32(dst)), "l"(src) : "memory");
}
// 4 bytes, or zeros when `valid` is false (nothing is read then; src is a valid address regardless)
__device__ __forceinline__ void cp_async4(float* dst, const void* src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(su32(dst)), "l"(src), "r"(valid ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// the 64 helper threads (warps 2 and 3)
__device__ __forceinline__ void helper_bar() { asm volatile("bar.sync 1, 64;" ::: "memory"); }
// the same barrier, returning whether `ok` holds for all 64 (one outcome for all)
__device__ __forceinline__ bool helper_all(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, 64, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"(ok ? 1u : 0u)
        : "memory");
    return r != 0;
}

// dst[0 .. n) = src[0 .. n) (32-bit elements), elements at index >= valid zero
// filled; 16-byte copies when the whole run is valid and aligned.  ht: helper thread 0..63.
__device__ __forceinline__ void side_copy(float* dst, const void* src, int n, int64_t valid, int ht) {
    const char* s = static_cast<const char*>(src);
    if (valid >= n && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
        for (int i = 4 * ht; i < n; i += 4 * 64) cp_async16(dst + i, s + 4 * (size_t)i);
    } else {
        for (int i = ht; i < n; i += 64) cp_async4(dst + i, i < valid ? s + 4 * (size_t)i : s, i < valid);
    }
}

// Copies and converts the side data of one tile (rows m0 .., columns n0 .. of
// problem P) into `sd`.  All 64 helper threads call it; it ends with their
// shared barrier passed, so every value is in place when they arrive.
// Rounds of side data a tile takes: the dW two-way correction stages kBch
// examples per round; everything else fits one.
__device__ __forceinline__ int side_rounds(const Problem& P, bool dw) {
    if (!dw || P.ec_mode != S3R_EC_TWO_WAY || P.B <= kBch) return 1;
    return (int)((P.B + kBch - 1) / kBch);
}

// The row threshold of token t under the glue's rounding (as the quantizers draw it).
__device__ __forceinline__ float glue_threshold(const Glue& G, uint64_t t, uint32_t tid) {
    if (G.thr == 1) return token_threshold7(t, G.seed_lo, tid);
    if (G.thr == 2) return example_threshold(G.S > 0 ? t / (uint64_t)G.S : 0u, G.seed_lo, tid);
    return token_threshold(t, G.seed_lo, tid);
}

// G: the glue of this tile's problem, or null.
template <int KIND>
__device__ __forceinline__ void load_side(const Problem& P, float* sd, int64_t m0, int64_t n0, int ht, int round,
                                          const Glue* G) {
    const int64_t rows = P.M - m0 < BM ? P.M - m0 : BM;      // valid rows of the tile
    const int64_t cols = P.N - n0 < BN ? P.N - n0 : BN;      // valid columns
    if (KIND == kDX) {
        if (P.s_row) side_copy(sd + SX_ROWSC, P.s_row + m0, BM, rows, ht);
        const int nseg = P.seg[1].K > 0 ? 2 : 1;
        int64_t b_lo = 0, b_hi = 0;
        if (P.ec_mode) {
            b_lo = m0 / P.S;
            b_hi = (m0 + rows - 1) / P.S;
            for (int g = 0; g < nseg; ++g) {
                side_copy(sd + SX_EPS + g * 128, P.seg[g].eps + m0, BM, rows, ht);
                side_copy(sd + SX_RS + g * 256, P.seg[g].rowsum + n0, BN, cols, ht);
                for (int64_t i = 0; i < kNbX && b_lo + i <= b_hi; ++i)
                    side_copy(sd + SX_V + (g * kNbX + (int)i) * 256, P.seg[g].v + (b_lo + i) * P.N + n0, BN, cols, ht);
            }
        }
        if (G) {
            if (G->s_x) side_copy(sd + SG_SX, G->s_x + m0, BM, rows, ht);
            if (G->s_w1) side_copy(sd + SG_SW1, G->s_w1 + n0, BN, cols, ht);
            if (G->s_w3) side_copy(sd + SG_SW3, G->s_w3 + n0, BN, cols, ht);
        }
        cp_async_wait_all();
        helper_bar();
        if (G) {
            if (!G->s_x)
                for (int i = ht; i < BM; i += 64) sd[SG_SX + i] = 1.0f;
            for (int j = ht; j < BN; j += 64) {
                if (!G->s_w1) sd[SG_SW1 + j] = 1.0f;
                if (!G->s_w3) sd[SG_SW3 + j] = 1.0f;
            }
        }
        for (int i = ht; i < BM; i += 64)
            sd[SX_ROWSC + i] = P.s_row ? __frcp_rn(sd[SX_ROWSC + i]) : 1.0f;   // 1/s of a zero-filled row is unused
        if (P.ec_mode) {
            for (int g = 0; g < 2; ++g) {
                for (int j = ht; j < BN; j += 64)
                    sd[SX_RS + g * 256 + j] = g < nseg ? (float)__float_as_int(sd[SX_RS + g * 256 + j]) : 0.0f;
                if (g >= nseg)
                    for (int i = ht; i < BM; i += 64) sd[SX_EPS + g * 128 + i] = 0.0f;
            }
        }
    } else {
        const bool two = P.ec_mode == S3R_EC_TWO_WAY;
        const int64_t b0 = (int64_t)round * kBch;
        const int nb = two ? (int)(P.B - b0 < kBch ? P.B - b0 : kBch) : 0;
        if (round == 0) {
            if (P.s_col) side_copy(sd + SW_COLSC, P.s_col + n0, BN, cols, ht);
            if (two) side_copy(sd + SW_P, P.p + m0, BM, rows, ht);
        }
        for (int b = 0; b < nb; ++b) {
            side_copy(sd + SW_XS + b * 128, P.xsum + (b0 + b) * P.M + m0, BM, rows, ht);
            side_copy(sd + SW_CM + b * 256, P.colmean + (b0 + b) * P.N + n0, BN, cols, ht);
        }
        cp_async_wait_all();
        helper_bar();
        if (round == 0)
            for (int j = ht; j < BN; j += 64) sd[SW_COLSC + j] = P.s_col ? __frcp_rn(sd[SW_COLSC + j]) : 1.0f;
        for (int b = 0; b < nb; ++b) {
            const float mb = __ldg(P.mu + b0 + b);
            for (int i = ht; i < BM; i += 64) sd[SW_XS + b * 128 + i] = (float)__float_as_int(sd[SW_XS + b * 128 + i]);
            for (int j = ht; j < BN; j += 64) sd[SW_CM + b * 256 + j] = sd[SW_CM + b * 256 + j] - mb;
        }
    }
    helper_bar();
}

// Subtracts the correction (or, for dW, one round of it) from the thread's
// accumulators (row `row`, local row rl of the tile, its 128 columns of half
// `half`), from the side data:
//   dX: acc -= eps_g[t] rowsum_g[k] + v_g[t/S, k] for each term g;
//   dW: acc -= sum_b xsum[b, k] (colmean[b, n] - mu[b]) over the round's
//       examples, and p[k] in round 0 (two-way).
template <int KIND>
__device__ __forceinline__ void apply_correction(const Problem& P, float (&acc)[128], const float* sd, int64_t row,
                                                 int64_t m0, int rl, int half, int round) {
    if (KIND == kDX) {
        if (!P.ec_mode) return;
        const int i_row = row < P.M ? (int)(row / P.S - m0 / P.S) : 0;
        const int nseg = P.seg[1].K > 0 ? 2 : 1;
        for (int g = 0; g < nseg; ++g) {
            const float ep = sd[SX_EPS + g * 128 + rl];
            const float2 ep2 = make_float2(ep, ep);
            const float* rs = sd + SX_RS + g * 256 + 128 * half;
            const float* vv = sd + SX_V + (g * kNbX + i_row) * 256 + 128 * half;
#pragma unroll
            for (int j4 = 0; j4 < 128; j4 += 4) {
                const float4 r = lds4(rs + j4), w = lds4(vv + j4);
                const float2 a = f2_fma(ep2, make_float2(r.x, r.y), make_float2(w.x, w.y));
                const float2 b = f2_fma(ep2, make_float2(r.z, r.w), make_float2(w.z, w.w));
                const float2 x = f2_sub(make_float2(acc[j4], acc[j4 + 1]), a);
                const float2 y = f2_sub(make_float2(acc[j4 + 2], acc[j4 + 3]), b);
                acc[j4 + 0] = x.x;
                acc[j4 + 1] = x.y;
                acc[j4 + 2] = y.x;
                acc[j4 + 3] = y.y;
            }
        }
    } else {
        if (P.ec_mode != S3R_EC_TWO_WAY) return;
        const int64_t b0 = (int64_t)round * kBch;
        const int nb = (int)(P.B - b0 < kBch ? P.B - b0 : kBch);
        for (int b = 0; b < nb; ++b) {
            const float nx = -sd[SW_XS + b * 128 + rl];
            const float2 nx2 = make_float2(nx, nx);
            const float* cm = sd + SW_CM + b * 256 + 128 * half;
#pragma unroll
            for (int j4 = 0; j4 < 128; j4 += 4) {
                const float4 c4 = lds4(cm + j4);
                const float2 x = f2_fma(nx2, make_float2(c4.x, c4.y), make_float2(acc[j4], acc[j4 + 1]));
                const float2 y = f2_fma(nx2, make_float2(c4.z, c4.w), make_float2(acc[j4 + 2], acc[j4 + 3]));
                acc[j4 + 0] = x.x;
                acc[j4 + 1] = x.y;
                acc[j4 + 2] = y.x;
                acc[j4 + 3] = y.y;
            }
        }
        if (round) return;
        const float pr = sd[SW_P + rl];
        const float2 pr2 = make_float2(pr, pr);
#pragma unroll
        for (int j = 0; j < 128; j += 2) {
            const float2 x = f2_sub(make_float2(acc[j], acc[j + 1]), pr2);
            acc[j] = x.x;
            acc[j + 1] = x.y;
        }
    }
}

// The final rescale: times 1/s_x[t] (dX) or 1/s_w[n] (dW), from the side data.
template <int KIND>
__device__ __forceinline__ void rescale(const Problem& P, float (&acc)[128], const float* sd, int rl, int half) {
    if (KIND == kDX) {
        if (!P.s_row) return;
        const float r = sd[SX_ROWSC + rl];
        const float2 r2 = make_float2(r, r);
#pragma unroll
        for (int j = 0; j < 128; j += 2) {
            const float2 x = f2_mul(make_float2(acc[j], acc[j + 1]), r2);
            acc[j] = x.x;
            acc[j + 1] = x.y;
        }
    } else {
        if (!P.s_col) return;
        const float* cs = sd + SW_COLSC + 128 * half;
#pragma unroll
        for (int j4 = 0; j4 < 128; j4 += 4) {
            const float4 r = lds4(cs + j4);
            const float2 x = f2_mul(make_float2(acc[j4], acc[j4 + 1]), make_float2(r.x, r.y));
            const float2 y = f2_mul(make_float2(acc[j4 + 2], acc[j4 + 3]), make_float2(r.z, r.w));
            acc[j4 + 0] = x.x;
            acc[j4 + 1] = x.y;
            acc[j4 + 2] = y.x;
            acc[j4 + 3] = y.y;
        }
    }
}

// Forward scaling: the exact int32 sum converted once, then (acc * s_x[row]) *
// s_w[col], one rounding each; columns past N are scaled by 1.
__device__ __forceinline__ void fwd_scale(const Problem& P, float (&acc)[128], int64_t row, int64_t c0) {
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

// ---------------------------------------------------------------------------
// Output: the warp's 32 rows x 128 columns (thread = row) leave through the
// TMA engine, 8 columns per bulk store: each lane writes its row of 32 bytes
// into a staging buffer in the 32-byte swizzled layout of the tensor map (the
// second 16-byte half first on rows 4..7 of every 8), so the writes are free
// of bank conflicts; lane 0 then issues the store (or an add-reduction when
// the result accumulates into C).  The TMA engine drops what lies outside C.
// Two buffers per warp alternate; a buffer is rewritten only after the store
// that read it has finished reading (bulk async-group wait).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void tma_store(const CUtensorMap* map, uint32_t src, int32_t x, int32_t y, bool add) {
    if (add)
        asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                         (uint64_t)map),
                     "r"(x), "r"(y), "r"(src)
                     : "memory");
    else
        asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"((uint64_t)map),
                     "r"(x), "r"(y), "r"(src)
                     : "memory");
}

// x0: first column of the thread's 128; y0 = row - lane: first row of the warp's 32.
__device__ __forceinline__ void store_tile(const Problem& P, const CUtensorMap* cmap, const float (&acc)[128],
                                           uint8_t* obuf, int64_t row, int64_t x0, int lane) {
    const bool accum = P.accumulate != 0;
    if (P.c_tma) {
        const int64_t y0 = row - lane;
        const int sw = (lane >> 2) & 1;
#pragma unroll
        for (int c = 0; c < 128 / OUT_COLS; ++c) {
            uint8_t* b = obuf + (c & 1) * OUT_BUF_BYTES;
            if (lane == 0) bulk_wait_read1();   // the store that last read b has read it
            __syncwarp();
            float4* r = reinterpret_cast<float4*>(b + lane * 32);
            r[sw] = make_float4(acc[8 * c + 0], acc[8 * c + 1], acc[8 * c + 2], acc[8 * c + 3]);
            r[sw ^ 1] = make_float4(acc[8 * c + 4], acc[8 * c + 5], acc[8 * c + 6], acc[8 * c + 7]);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                const int64_t x = x0 + OUT_COLS * c;
                if (x < P.N && y0 < P.M) tma_store(cmap, su32(b), (int32_t)x, (int32_t)y0, accum);
                bulk_commit();
            }
        }
    } else if (row < P.M) {   // C not addressable by the TMA engine: plain stores
        float* dst = P.C + row * P.ldc + x0;
#pragma unroll
        for (int j = 0; j < 128; ++j)
            if (x0 + j < P.N) dst[j] = accum ? dst[j] + acc[j] : acc[j];
    }
}

// ---------------------------------------------------------------------------
// The SwiGLU glue epilogue (kMixedG launches, the glue problem's tiles).  A
// warpgroup's 128 rows x 128 columns of dA (thread = row, acc after the
// correction and the 1/s_x rescale) are exactly one 128 x 128 tile of dh1
// and of dh3, so the whole quantization of both happens here:
//   pass 1: h1, h3 of the thread's row (16-byte loads, prefetched to L2 a few
//           blocks earlier), the glue and the folds in the order of the
//           separate SwiGLU quantizer (two lanes per packed instruction);
//           the folded dh1 replaces dA in acc, the folded dh3 goes into the
//           tile's own TMEM accumulator (still held back from the MMA
//           issuer), and the two absmaxes meet across the warpgroup;
//   pass 2: per output the tile scale, the codes (16-byte stores of fp16
//           codes), the per-token error sum of the row and the per-channel
//           sums over the warp's 32 rows (a reduce-scatter), which meet
//           across the warpgroup in a fixed order through the warps' staging
//           buffers.
// The exchanges use three mbarriers per warpgroup (count 4, lane 0 of each
// warp), waited on with the bounded wait; returns false if one ran out.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// v[0..16): one value per column of a 16-column chunk, the thread's row.
// Returns the sum over the warp's 32 lanes (rows) of column (lane >> 1); the
// pairs are added in a fixed order (halving exchanges on lane bits 4..1,
// then bit 0).
__device__ __forceinline__ float colsum16(const float (&v)[16], int lane) {
    float a[8], b[4], c[2];
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = (b4 ? v[i + 8] : v[i]) + __shfl_xor_sync(0xFFFFFFFFu, b4 ? v[i] : v[i + 8], 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) b[i] = (b3 ? a[i + 4] : a[i]) + __shfl_xor_sync(0xFFFFFFFFu, b3 ? a[i] : a[i + 4], 8);
#pragma unroll
    for (int i = 0; i < 2; ++i) c[i] = (b2 ? b[i + 2] : b[i]) + __shfl_xor_sync(0xFFFFFFFFu, b2 ? b[i] : b[i + 2], 4);
    float d = (b1 ? c[1] : c[0]) + __shfl_xor_sync(0xFFFFFFFFu, b1 ? c[0] : c[1], 2);
    d += __shfl_xor_sync(0xFFFFFFFFu, d, 1);
    return d;
}

// Rounds the folded values in acc (the thread's row, columns c0 ..) to codes
// with step d and normalizer inv, stores them (fp16) into Q and the error
// partials: returns the row's sum of g - d q; the warp's column sums of it go
// to xc[0..128).
__device__ __forceinline__ float glue_round(const Glue& G, const float (&acc)[128], float d, float inv, bool nonfinite,
                                            float u, bool vrow, int64_t row, int64_t c0, int64_t F, uint16_t* Q,
                                            bool err, float* xc, int lane) {
    const float2 M2 = make_float2(kMagic, kMagic), inv2 = make_float2(inv, inv), nd2 = make_float2(-d, -d);
    const float2 uu = make_float2(u, u);
    float2 rs = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
        float ne[16];
        uint32_t hw[8];
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
            const float2 g2 = make_float2(acc[16 * cc + i], acc[16 * cc + i + 1]);
            float2 qq = make_float2(0.0f, 0.0f), e = make_float2(0.0f, 0.0f);
            if (!nonfinite) {
                const float2 y = f2_mul(g2, inv2);   // |y| <= 127
                float2 m;
                if (G.rtne)   // per lane: a packed add that is the product's only use would be fused into an fma
                    m = make_float2(__fadd_rn(y.x, kMagic), __fadd_rn(y.y, kMagic));
                else
                    m = f2_add_rp(f2_sub_rp(y, uu), M2);   // kMagic + ceil(y - u) = kMagic + floor(y) + [u < frac(y)]
                qq = f2_sub(m, M2);
                e = f2_fma(nd2, qq, g2);   // g - delta q
            }
            ne[i] = e.x;
            ne[i + 1] = e.y;
            rs = f2_add(rs, e);
            const __half2 h2 = __floats2half2_rn(qq.x, qq.y);
            hw[i / 2] = *reinterpret_cast<const uint32_t*>(&h2);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t col = c0 + 16 * cc + 8 * h;
            if (vrow && col < F)
                *reinterpret_cast<uint4*>(Q + row * F + col) = make_uint4(hw[4 * h], hw[4 * h + 1], hw[4 * h + 2],
                                                                          hw[4 * h + 3]);
        }
        if (err) {
            const float cs = colsum16(ne, lane);
            if ((lane & 1) == 0) xc[16 * cc + (lane >> 1)] = cs;
        }
    }
    return rs.x + rs.y;
}

// tcol: TMEM address of the thread's lane, its 128 columns, in the tile's last
// accumulator; xbase: the staging area of this warpgroup's four warps (2 KiB
// each, as float[2][128] for the column exchange); gam: absmax exchange
// [warp][output]; ph: glue tiles this warpgroup has finished.
__device__ __forceinline__ bool glue_tile(const Glue& G, const Problem& P, float (&acc)[128], const float* sd,
                                          uint32_t tcol, int64_t row, int rl, int64_t mt, int64_t nt, int64_t c0,
                                          int half, int q, int lane, uint8_t* xbase, uint32_t (*gam)[2],
                                          uint32_t barA, uint32_t barB, uint32_t barC, uint32_t ph,
                                          volatile int* abrt, int* d_status) {
    const int64_t F = P.N;
    const bool vrow = row < P.M;
    const float sx = sd[SG_SX + rl];
    const float2 sx2 = make_float2(sx, sx);
    const float* sw1 = sd + SG_SW1 + 128 * half;
    const float* sw3 = sd + SG_SW3 + 128 * half;
    const uint16_t* p1 = G.h1 + row * G.ldh + c0;   // read only for valid rows and columns
    const uint16_t* p3 = G.h3 + row * G.ldh + c0;
    // ---- pass 1: glue, folds, absmax; dh1 into acc, dh3 into TMEM (8 columns at a time) ----
    float am1 = 0.0f, am3 = 0.0f;   // NaN-propagating
#pragma unroll
    for (int cc = 0; cc < 16; ++cc) {
        const bool okg = vrow && c0 + 8 * cc < F;
        uint4 a = make_uint4(0u, 0u, 0u, 0u), b = make_uint4(0u, 0u, 0u, 0u);
        if (okg) {
            a = __ldg(reinterpret_cast<const uint4*>(p1 + 8 * cc));
            b = __ldg(reinterpret_cast<const uint4*>(p3 + 8 * cc));
        }
        const uint32_t w1[4] = {a.x, a.y, a.z, a.w}, w3[4] = {b.x, b.y, b.z, b.w};
        uint32_t v3[8];
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            const int j = 8 * cc + i;
            // glue, in the documented order, two lanes per packed instruction
            // (no contraction: built with -fmad=false)
            const float2 x = make_float2(bf16_lo(w1[i >> 1]), bf16_hi(w1[i >> 1]));
            const float2 x3 = make_float2(bf16_lo(w3[i >> 1]), bf16_hi(w3[i >> 1]));
            const float2 d2 = okg ? make_float2(acc[j], acc[j + 1]) : make_float2(0.0f, 0.0f);
            float2 silu, dsilu;
            swiglu_terms2(x, silu, dsilu);
            const float2 dh1 = f2_mul(f2_mul(d2, x3), dsilu);
            const float2 dh3 = f2_mul(d2, silu);
            // folds (s_x * dh) * s_w
            const float2 g1 = f2_mul(f2_mul(sx2, dh1), make_float2(sw1[j], sw1[j + 1]));
            const float2 g3 = f2_mul(f2_mul(sx2, dh3), make_float2(sw3[j], sw3[j + 1]));
            acc[j] = g1.x;
            acc[j + 1] = g1.y;
            v3[i] = __float_as_uint(g3.x);
            v3[i + 1] = __float_as_uint(g3.y);
            am1 = max3_abs_nan(am1, g1.x, g1.y);
            am3 = max3_abs_nan(am3, g3.x, g3.y);
        }
        tmem_st8(tcol + 8 * cc, v3);
    }
    tmem_wait_st();   // the loads of pass 2 read what these stores wrote
    {
        const uint32_t m1 = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(am1));
        const uint32_t m3 = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(am3));
        if (lane == 0) {
            gam[q][0] = m1;
            gam[q][1] = m3;
        }
    }
    // the column exchange reuses the warp's staging buffers: the stores that read them are done first
    if (lane == 0) bulk_wait_read0();
    __syncwarp();
    if (lane == 0) mbar_arrive(barA);
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(barA, ph & 1u, abrt))) return false;
    const uint32_t amax1 = max(max(gam[0][0], gam[1][0]), max(gam[2][0], gam[3][0]));
    const uint32_t amax3 = max(max(gam[0][1], gam[1][1]), max(gam[2][1], gam[3][1]));
    float d1, inv1, d3, inv3;
    tile_scales(amax1, d1, inv1);
    tile_scales(amax3, d3, inv3);
    const bool nf1 = amax1 >= 0x7F800000u, nf3 = amax3 >= 0x7F800000u;
    if (q == 0 && lane == 0) {
        G.scale1[mt * G.ntc + nt] = d1;
        G.scale3[mt * G.ntc + nt] = d3;
        if (nf1 || nf3) set_status(d_status, S3R_ERR_NONFINITE);
    }
    // ---- pass 2: codes and error partials, dh1 from acc, then dh3 from TMEM ----
    const bool err = G.tok1 != nullptr;
    float* xc = reinterpret_cast<float*>(xbase + q * (2 * OUT_BUF_BYTES));   // this warp's [2][128]
    // the row's thresholds (one Philox draw each, as the quantizers draw them)
    const float u1 = G.rtne ? 0.0f : glue_threshold(G, (uint64_t)row, G.tid1);
    const float u3 = G.rtne ? 0.0f : glue_threshold(G, (uint64_t)row, G.tid3);
    const float r1 = glue_round(G, acc, d1, inv1, nf1, u1, vrow, row, c0, F, G.Q1, err, xc, lane);
#pragma unroll
    for (int c = 0; c < 8; c += 4) {
        uint32_t r[4][16];
#pragma unroll
        for (int u = 0; u < 4; ++u) tmem_ld16(tcol + 16 * (c + u), r[u]);
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[16 * (c + u) + j] = __uint_as_float(r[u][j]);
    }
    const float r3 = glue_round(G, acc, d3, inv3, nf3, u3, vrow, row, c0, F, G.Q3, err, xc + 128, lane);
    if (err && vrow) {
        G.tok1[row * G.ntc + nt] = -r1;
        G.tok3[row * G.ntc + nt] = -r3;
    }
    if (err) {
        __syncwarp();
        if (lane == 0) mbar_arrive(barB);
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(barB, ph & 1u, abrt))) return false;
        // thread 32 q + lane adds its column over the four warps, in warp order
        const int tix = 32 * q + lane;
        if (c0 + tix < F) {
            float s1 = 0.0f, s3 = 0.0f;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float* xw = reinterpret_cast<const float*>(xbase + w * (2 * OUT_BUF_BYTES));
                s1 += xw[tix];
                s3 += xw[128 + tix];
            }
            G.col1[mt * F + c0 + tix] = -s1;
            G.col3[mt * F + c0 + tix] = -s3;
        }
        // every warp has read the staging buffers before any of them is written again
        __syncwarp();
        if (lane == 0) mbar_arrive(barC);
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(barC, ph & 1u, abrt))) return false;
    }
    return true;
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

// The next tile of CTA b (of G) in the launch: problems in order, within a
// problem the CTA's tiles of the deal (Args::deal_s) in increasing
// order.  (p, k): the caller's position, zero-initialized.  Every role of the
// CTA walks the same sequence.
__device__ __forceinline__ bool next_tile(const Args& A, int b, int G, int& p, int& k, int& tile) {
    while (p < A.nprob) {
        const Problem& P = A.prob[p];
        int t;
        if (deal::kth_tile(P.ntm * P.ntn, A.deal_s[p], A.deal_w[p], A.deal_m[p], b, G, k, t)) {
            tile = P.tile_base + t;
            ++k;
            return true;
        }
        ++p;
        k = 0;
    }
    return false;
}

// The launch problem that owns launch tile `tile` (tiles of problem i start at
// prob[i].tile_base, in increasing order).
__device__ __forceinline__ int problem_of(const Args& A, int tile) {
    int i = 0;
    while (i + 1 < A.nprob && tile >= A.prob[i + 1].tile_base) ++i;
    return i;
}

// A CTA's walk over its tiles, as launch tile indices (ntiles: past the last).
// Mixed launches (problems with tiles of different lengths) walk the host's
// deal, (p, k) holding the current tile's problem and its place in the deal;
// the others, whose deal is plain round robin, step the index by the grid.
template <bool DEAL>
__device__ __forceinline__ int first_tile(const Args& A, int ntiles, int& p, int& k) {
    if constexpr (DEAL) {
        int t;
        return next_tile(A, (int)blockIdx.x, (int)gridDim.x, p, k, t) ? t : ntiles;
    } else {
        return (int)blockIdx.x;
    }
}
template <bool DEAL>
__device__ __forceinline__ int following_tile(const Args& A, int ntiles, int& p, int& k, int tile) {
    if constexpr (DEAL) {
        int t;
        return next_tile(A, (int)blockIdx.x, (int)gridDim.x, p, k, t) ? t : ntiles;
    } else {
        return tile + (int)gridDim.x;
    }
}
// The problem of the walk's current tile.
template <bool DEAL>
__device__ __forceinline__ int tile_problem(const Args& A, int p, int tile) {
    if constexpr (DEAL) return p;
    else return problem_of(A, tile);
}

// 12 warps: one SM sub-partition hosts three of them, one per warpgroup, so the
// launch is capped at 168 registers per thread; after the split a
// sub-partition holds (56 + 216 + 216) * 32 = 15616 of its 16384.
template <int EPI, bool MN>
__global__ void __launch_bounds__(THREADS, 1)
    umma_gemm_kernel(const __grid_constant__ Maps maps, const __grid_constant__ Args A) {
    // the side-data protocol (helper warps, correction inside the tile) serves the backward kinds
    constexpr bool SIDE = EPI == kDX || EPI == kDW || EPI == kMixed || EPI == kMixedG;
    constexpr bool MIXED = EPI == kMixed || EPI == kMixedG;   // each problem has its own kind (kDX or kDW)
    extern __shared__ uint8_t smem_raw[];
    __shared__ int abort_flag;
    __shared__ uint32_t glue_amax[2][4][2];   // glue epilogue: absmax exchange [warpgroup][warp][output]
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_STAGE;
    uint8_t* sOut = sB + STAGES * B_STAGE;   // 1024-byte aligned: the swizzle atoms start on it
    float* sSide = reinterpret_cast<float*>(sOut + OUT_STAGE_BYTES);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sSide + SIDE_FLOATS);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
    const uint32_t full0 = su32(bars), empty0 = su32(bars + STAGES), tfull0 = su32(bars + 2 * STAGES),
                   tempty0 = su32(bars + 2 * STAGES + 2), done_bar = su32(bars + 2 * STAGES + 4),
                   side_full = su32(bars + 2 * STAGES + 5), side_empty = su32(bars + 2 * STAGES + 6),
                   glue_bar0 = su32(bars + 2 * STAGES + 7);   // [A, B, C] x [warpgroup]

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
        mbar_init(side_full, 64);          // the 64 helper threads
        mbar_init(side_empty, EPI_WARPS);  // lane 0 of each epilogue warp
        for (int b = 0; b < 6; ++b) mbar_init(glue_bar0 + 8 * b, 4);   // lane 0 of each warp of a warpgroup
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

    // Persistent: this CTA walks the tiles the host's deal gives it (next_tile).
    // The smem ring and the TMEM double buffer keep their phases across tiles,
    // so the next tile's copies and MMAs start while the epilogue still stores
    // the previous tile.
    if (warp < EPI_WARP0) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(EPI == kMixedG ? kRegsLowGlue : kRegsLow));
        if (warp == 0) {
            if (lane == 0) {
                int it = 0;   // slice counter over the whole persistent run
                int last_pi = -1;
                bool ok = true;
                int sp = 0, sk = 0;
                for (int tile = first_tile<MIXED>(A, ntiles, sp, sk); tile < ntiles && ok;
                     tile = following_tile<MIXED>(A, ntiles, sp, sk, tile)) {
                    const int pi = tile_problem<MIXED>(A, sp, tile);
                    const Problem& P = A.prob[pi];
                    const CUtensorMap* mp = &maps.m[pi][0];
                    const int nkb0 = (int)s3r_cdiv(P.seg[0].K, 128), nkb1 = (int)s3r_cdiv(P.seg[1].K, 128);
                    const int nkb = nkb0 + nkb1;   // 128-wide blocks of this tile
                    if (pi != last_pi) {
                        for (int j = 0; j < (nkb1 || (EPI == kFwdE && P.kind == kGate) || (EPI == kMixedG && pi == A.glue.prob)
                                                 ? 4 : 2); ++j)
                            asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)(mp + j)) : "memory");
                        last_pi = pi;
                    }
                    int tm, tn;
                    tile_coords(tile - P.tile_base, P.ntm, P.ntn, P.band_rows, tm, tn);
                    const bool gate = EPI == kFwdE && P.kind == kGate;
                    const int32_t m0 = tm * BM, n0 = tn * (gate ? BN / 2 : BN);
                    // glue tile: its h1 and h3 boxes into L2 a few blocks before the tile ends
                    // (maps 2 and 3 of the one-term glue problem)
                    const int pf_sl = EPI == kMixedG && pi == A.glue.prob ? 2 * (nkb > 4 ? nkb - 4 : 0) : -1;
                    for (int sl = 0; sl < 2 * nkb; ++sl, ++it) {
                        if (sl == pf_sl) {
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];" ::"l"(
                                                 (uint64_t)(mp + 2 + (j >> 2))),
                                             "r"(n0 + 64 * (j & 3)), "r"(m0)
                                             : "memory");
                        }
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
                        const bool a_mn = MIXED ? P.kind == kDW : (EPI == kFwdE ? false : MN);
                        const bool b_mn = MIXED ? P.kind == kDW : (EPI == kFwdE ? true : MN);
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
                int sp = 0, sk = 0;
                for (int tile = first_tile<MIXED>(A, ntiles, sp, sk); tile < ntiles && ok;
                     tile = following_tile<MIXED>(A, ntiles, sp, sk, tile)) {
                    const Problem& P = A.prob[tile_problem<MIXED>(A, sp, tile)];
                    const int nkb = (int)(s3r_cdiv(P.seg[0].K, 128) + s3r_cdiv(P.seg[1].K, 128));
                    const bool a_mn = MIXED ? P.kind == kDW : (EPI == kFwdE ? false : MN);
                    const bool b_mn = MIXED ? P.kind == kDW : (EPI == kFwdE ? true : MN);
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
        } else if (SIDE) {
            // ------------------------------ helpers (warps 2, 3) ------------------------------
            // Bring each tile's epilogue vectors into the side buffer as soon as the
            // epilogue has finished with the previous tile's.
            const int ht = threadIdx.x - 64;
            uint32_t sph = 0;   // side-buffer cycles so far (the same count on the epilogue side)
            bool ok = true;
            int sp = 0, sk = 0;
            for (int tile = first_tile<MIXED>(A, ntiles, sp, sk); tile < ntiles && ok;
                 tile = following_tile<MIXED>(A, ntiles, sp, sk, tile)) {
                const Problem& P = A.prob[tile_problem<MIXED>(A, sp, tile)];
                int tm, tn;
                tile_coords(tile - P.tile_base, P.ntm, P.ntn, P.band_rows, tm, tn);
                const int64_t m0 = (int64_t)tm * BM, n0 = (int64_t)tn * BN;
                const bool dw = MIXED ? P.kind == kDW : EPI == kDW;
                const int nr = side_rounds(P, dw);
                for (int r = 0; r < nr; ++r, ++sph) {
                    // one outcome for both helper warps: they meet at named barriers below
                    if (!helper_all(mbar_wait(side_empty, (sph & 1u) ^ 1u, abrt))) {
                        *abrt = 1;
                        ok = false;
                        break;
                    }
                    const Glue* G = (EPI == kMixedG && tile_problem<MIXED>(A, sp, tile) == A.glue.prob) ? &A.glue : nullptr;
                    if (dw) load_side<kDW>(P, sSide, m0, n0, ht, r, nullptr);
                    else load_side<kDX>(P, sSide, m0, n0, ht, r, G);
                    mbar_arrive(side_full);
                }
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
        // ------------------------------ epilogue ------------------------------
        // warp w reads TMEM lanes 32 * (w % 4) ..; two warps per lane quarter
        // split the 256 accumulator columns into halves
        const int q = warp & 3, ew = warp - EPI_WARP0, half = ew >> 2;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
        uint8_t* obuf = sOut + ew * (2 * OUT_BUF_BYTES);
        const int rl = 32 * q + lane;   // row within the tile
        int gkb = 0;
        uint32_t sph = 0;   // side-buffer cycles so far (the same count on the helper side)
        uint32_t gph = 0;   // glue tiles this warpgroup has finished (phase of its exchange barriers)
        bool ok = true;
        int sp = 0, sk = 0;
        for (int tile = first_tile<MIXED>(A, ntiles, sp, sk); tile < ntiles && ok;
             tile = following_tile<MIXED>(A, ntiles, sp, sk, tile)) {
            const int pi = tile_problem<MIXED>(A, sp, tile);
            const Problem& P = A.prob[pi];
            const int nkb0 = (int)s3r_cdiv(P.seg[0].K, 128), nkb1 = (int)s3r_cdiv(P.seg[1].K, 128);
            const int nkb = nkb0 + nkb1;
            int tm, tn;
            tile_coords(tile - P.tile_base, P.ntm, P.ntn, P.band_rows, tm, tn);
            const int mt = tm, nt = tn * 2 + half;   // 128-wide tile indices
            const int64_t m0 = (int64_t)mt * BM;
            const int64_t row = m0 + rl;
            const bool gate = EPI == kFwdE && P.kind == kGate;
            const bool is_dw = MIXED ? P.kind == kDW : EPI == kDW;
            // glue tile: the last block's accumulator is held back from the MMA
            // issuer until the glue has used it for dh3
            const bool glue = EPI == kMixedG && pi == A.glue.prob;
            // gate: this half owns output columns c0 .. c0 + 63, accumulators
            // 0..63 = h1 (TMEM columns 64 half ..), 64..127 = h3 (128 + 64 half ..)
            const int64_t c0 = gate ? (int64_t)tn * 128 + 64 * half : (int64_t)nt * 128;
            const uint32_t col_base = (uint32_t)(gate ? 64 * half : 128 * half);
            const uint32_t col_step = gate ? 128u - 64u : 0u;   // extra offset of chunks 4..7
            float acc[128];
#pragma unroll
            for (int j = 0; j < 128; ++j) acc[j] = 0.0f;   // (int32 zero for the forward)
            // the correction enters after block kc (all its rounds); the last
            // round's side data stays for the final rescale
            const int kc = nkb - 1 < kCorrBlock ? nkb - 1 : kCorrBlock;
            const int nr = SIDE ? side_rounds(P, is_dw) : 0;
            auto correct = [&]() -> bool {
                for (int r = 0; r < nr; ++r) {
                    if (!__all_sync(0xFFFFFFFFu, mbar_wait(side_full, sph & 1u, abrt))) return false;
                    if (is_dw) apply_correction<kDW>(P, acc, sSide, row, m0, rl, half, r);
                    else apply_correction<kDX>(P, acc, sSide, row, m0, rl, half, r);
                    if (r + 1 < nr) {   // hand the buffer back for the next round
                        __syncwarp();
                        if (lane == 0) mbar_arrive(side_empty);
                        ++sph;
                    }
                }
                return true;
            };
            // scale of block kb, loaded one block ahead
            auto scale_of = [&](int kb) -> float {
                if (EPI == kDump) return 0.0f;
                const bool first = kb < nkb0;
                const int64_t kk = first ? kb : kb - nkb0;
                const float* base = first ? P.seg[0].scale : P.seg[1].scale;
                const int64_t off = first ? mt * P.seg[0].sm + nt * P.seg[0].sn + kk * P.seg[0].sk
                                          : mt * P.seg[1].sm + nt * P.seg[1].sn + kk * P.seg[1].sk;
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
                if (lane == 0 && !(glue && kb + 1 == nun)) mbar_arrive(tempty0 + 8 * buf);
                if (SIDE && kb == kc && !correct()) {   // after the TMEM hand-back: the MMA runs on meanwhile
                    ok = false;
                    *abrt = 1;
                    break;
                }
            }
            if (EPI == kDump || !ok) continue;
            if (SIDE) {
                if (nkb == 0 && !correct()) {   // no block ran: the correction alone
                    ok = false;
                    *abrt = 1;
                    continue;
                }
                if (is_dw) rescale<kDW>(P, acc, sSide, rl, half);
                else rescale<kDX>(P, acc, sSide, rl, half);
                if (EPI == kMixedG && glue) {
                    // acc is this warpgroup's 128 x 128 tile of dA: the glue and both quantizations
                    const uint32_t lb = (uint32_t)((gkb - 1) & 1);   // the held accumulator
                    if (c0 < P.N) {
                        if (!glue_tile(A.glue, P, acc, sSide, lane_addr + lb * BN + col_base, row, rl, mt, nt, c0,
                                       half, q, lane, sOut + (4 * half) * (2 * OUT_BUF_BYTES), glue_amax[half],
                                       glue_bar0 + 8 * half, glue_bar0 + 8 * (2 + half), glue_bar0 + 8 * (4 + half),
                                       gph, abrt, A.d_status)) {
                            ok = false;
                            *abrt = 1;
                            continue;
                        }
                        ++gph;
                    }
                    tmem_wait_st();
                    tc_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(tempty0 + 8 * lb);   // the accumulator goes back to the MMA issuer
                        mbar_arrive(side_empty);
                    }
                    ++sph;
                    continue;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(side_empty);   // the helpers may refill the side buffer
                ++sph;
                store_tile(P, &maps.m[pi][4], acc, obuf, row, c0, lane);
            } else if (EPI == kFwdE) {
                if (gate) {
                    finish_gate(P, acc, row, c0);
                } else {
                    fwd_scale(P, acc, row, c0);
                    store_tile(P, &maps.m[pi][4], acc, obuf, row, c0, lane);
                }
            }
        }
        // every bulk store has finished before the CTA (and its staging buffers) goes away
        if (lane == 0) bulk_wait_all();
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

// The output C [rows, cols] fp32 (row stride ldc elements) for the TMA stores
// of the epilogue: box 8 columns x 32 rows, 32-byte swizzle.  Leaves
// P.c_tma = 0 (plain stores) when C cannot be described (row stride or base
// not 16-byte aligned).
static int make_out_map(CUtensorMap* m, Problem& P) {
    P.c_tma = 0;
    if (!P.C || P.M <= 0 || P.N <= 0 || P.ldc % 4 != 0 || (reinterpret_cast<uintptr_t>(P.C) & 15u) != 0)
        return S3R_OK;
    auto fn = encode_fn();
    if (!fn) return S3R_ERR_CUDA;
    cuuint64_t dims[2] = {(cuuint64_t)P.N, (cuuint64_t)P.M};
    cuuint64_t strides[1] = {(cuuint64_t)P.ldc * 4};
    cuuint32_t box[2] = {(cuuint32_t)OUT_COLS, 32u};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, P.C, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char buf[200];
        snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled returned %d for the output (%lld x %lld, stride %lld)",
                 (int)r, (long long)P.M, (long long)P.N, (long long)P.ldc);
        s3r_record_error("tensor map", buf);
        return S3R_ERR_CUDA;
    }
    P.c_tma = 1;
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
    if (EPI == kMixed || EPI == kMixedG) {
        // the static deal of a mixed launch: a tile costs its 128-wide blocks plus about six
        // blocks' worth of tile end
        int64_t n[kMaxProb];
        double c[kMaxProb];
        deal::Plan plan[kMaxProb];
        for (int i = 0; i < A.nprob; ++i) {
            const Problem& P = A.prob[i];
            n[i] = (int64_t)P.ntm * P.ntn;
            c[i] = (double)(s3r_cdiv(P.seg[0].K, 128) + s3r_cdiv(P.seg[1].K, 128)) + 6.0;
        }
        deal::plan(A.nprob, n, c, (int)grid, plan);
        for (int i = 0; i < A.nprob; ++i) {
            A.deal_s[i] = plan[i].s;
            A.deal_w[i] = plan[i].w;
            A.deal_m[i] = plan[i].m;
        }
    } else {
        // the other kernels step the launch-wide tile index by the grid (walk<false>)
        for (int i = 0; i < A.nprob; ++i) {
            A.deal_s[i] = (int)(A.prob[i].tile_base % grid);
            A.deal_w[i] = (int)grid;
            A.deal_m[i] = 0;
        }
    }
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
    st = q.dump ? S3R_OK : umma::make_out_map(&m[4], P);
    if (st) return st;
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
    st = q.dump ? S3R_OK : umma::make_out_map(&m[4], P);
    if (st) return st;
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
    if (!gate) {
        st = umma::make_out_map(&m[4], P);
        if (st) return st;
    }
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

int umma_wait_probe(uint64_t limit_ns, int raise_abort, int* d_status, unsigned long long* waited_ns,
                    cudaStream_t stream) {
    umma::wait_probe_kernel<<<1, 64, 0, stream>>>(limit_ns, raise_abort, d_status, waited_ns);
    S3R_CHECK_LAUNCH();
    return S3R_OK;
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

// The glue of a kMixedG launch from its C-level description, for launch
// problem `prob` (a one-term dX problem of width F = P.N).
static int make_glue(umma::Glue& G, const UmmaGlue& g, const umma::Problem& P, int prob) {
    if (P.seg[1].K > 0) return S3R_ERR_ARG;   // dA has one contraction term
    const int64_t F = P.N;
    if (!g.h1 || !g.h3 || !g.Q1 || !g.Q3 || !g.scale1 || !g.scale3) return S3R_ERR_ARG;
    if ((g.tok1 == nullptr) != (g.col1 == nullptr) || (g.tok1 == nullptr) != (g.tok3 == nullptr) ||
        (g.tok3 == nullptr) != (g.col3 == nullptr))
        return S3R_ERR_ARG;
    if (g.ldh < F || F % 8 != 0 || g.ldh % 8 != 0 || !s3r_aligned16(g.h1) || !s3r_aligned16(g.h3) ||
        !s3r_aligned16(g.Q1) || !s3r_aligned16(g.Q3))
        return S3R_ERR_ALIGN;
    G = umma::Glue{};
    G.prob = prob;
    switch (g.round_mode) {
        case S3R_ROUND_S3R: G.thr = 0; break;
        case S3R_ROUND_S3R_7BIT: G.thr = 1; break;
        case S3R_ROUND_BCAST: G.thr = 2; break;
        case S3R_ROUND_RTNE: G.rtne = 1; break;
        default: return S3R_ERR_ARG;
    }
    if (G.rtne && g.tok1) return S3R_ERR_ARG;   // RTNE keeps no error partials
    G.seed_lo = (uint32_t)g.seed;
    G.tid1 = g.tid1;
    G.tid3 = g.tid3;
    G.S = g.S;
    G.h1 = static_cast<const uint16_t*>(g.h1);
    G.h3 = static_cast<const uint16_t*>(g.h3);
    G.ldh = g.ldh;
    G.s_x = g.s_x;
    G.s_w1 = g.s_w1;
    G.s_w3 = g.s_w3;
    G.Q1 = static_cast<uint16_t*>(g.Q1);
    G.Q3 = static_cast<uint16_t*>(g.Q3);
    G.scale1 = g.scale1;
    G.scale3 = g.scale3;
    G.tok1 = g.tok1;
    G.tok3 = g.tok3;
    G.col1 = g.col1;
    G.col3 = g.col3;
    G.ntc = s3r_cdiv(F, kTile);
    return S3R_OK;
}

// dX and dW problems in one launch (no dumps).  Problems run in the order of
// their per-tile contraction length, longest first, so the short tiles at the
// end of the round-robin fill in behind the long ones.  With a glue, dX
// problem glue->dx_index ends in the SwiGLU glue instead of a store.
static int mixed_group(const UmmaDxProblem* dx, int ndx, const UmmaDwProblem* dw, int ndw, const UmmaGlue* glue,
                       int* d_status, cudaStream_t stream) {
    const int n = ndx + ndw;
    if (ndx < 0 || ndw < 0 || n < 1 || n > umma::kMaxProb) return S3R_ERR_ARG;
    if (glue && (glue->dx_index < 0 || glue->dx_index >= ndx || dx[glue->dx_index].dX != nullptr ||
                 dx[glue->dx_index].accumulate))
        return S3R_ERR_ARG;
    thread_local umma::Maps maps;
    thread_local umma::Args A;
    std::memset(&A, 0, sizeof(A));
    A.glue.prob = -1;
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
        int st = i < ndx ? add_dx_problem(maps, A, k, dx[i], strip[k])
                         : add_dw_problem(maps, A, k, dw[i - ndx], strip[k]);
        if (!st && glue && i == glue->dx_index) {
            // maps 2 and 3 of the one-term glue problem describe h1 and h3 (L2 prefetches of the glue's boxes)
            st = make_glue(A.glue, *glue, A.prob[k], k);
            if (!st) st = umma::make_map(&maps.m[k][2], glue->h1, A.prob[k].N, A.prob[k].M, glue->ldh, umma::BM);
            if (!st) st = umma::make_map(&maps.m[k][3], glue->h3, A.prob[k].N, A.prob[k].M, glue->ldh, umma::BM);
        }
        if (st) return st;
    }
    A.nprob = n;
    A.d_status = d_status;
    if (glue) return umma::launch<umma::kMixedG, false>(maps, A, strip, stream);
    return umma::launch<umma::kMixed, false>(maps, A, strip, stream);
}

int umma_mixed_group(const UmmaDxProblem* dx, int ndx, const UmmaDwProblem* dw, int ndw, int* d_status,
                     cudaStream_t stream) {
    return mixed_group(dx, ndx, dw, ndw, nullptr, d_status, stream);
}

int umma_mixed_group_glue(const UmmaDxProblem* dx, int ndx, const UmmaDwProblem* dw, int ndw, const UmmaGlue* glue,
                          int* d_status, cudaStream_t stream) {
    if (!glue) return S3R_ERR_ARG;
    return mixed_group(dx, ndx, dw, ndw, glue, d_status, stream);
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
