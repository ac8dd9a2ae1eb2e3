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
// Kernel layout (one CTA per 128 x 256 output tile, 320 threads):
//   warp 0      TMA producer: 4-stage ring of 64-deep K slices in smem
//               (128-byte swizzle), one mbarrier pair per stage;
//   warp 1      allocates 512 TMEM columns; lane 0 issues tcgen05.mma
//               (M=128, N=256, K=16) into one of two 256-column fp32
//               accumulators (double buffer) and commits to mbarriers;
//   warps 2..9  epilogue: per 128-K block, tcgen05.ld their 32 TMEM lanes x
//               128 columns, acc = fma(scale, block, acc) in registers; at the
//               end apply the correction and the 1/s rescale and store fp32.
// Both products use the same kernel: dX reads K-major operands (Q [T,N] and
// W [K,N] contract over N); dW reads MN-major operands (X [T,K] and Q [T,N]
// contract over T), which the UMMA descriptors address directly.
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
constexpr int THREADS = 320;
constexpr uint32_t TMEM_COLS = 512;
constexpr int NUM_BARS = 2 * STAGES + 5;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + NUM_BARS * 8 + 16;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait

enum Epi { kDX = 0, kDW = 1, kDump = 2 };

struct Args {
    int64_t M, N, K;             // C[M, N] = sum_k A[m, k] B[n, k]
    const float* scale;          // scale(mt, nt, kb) = scale[mt*sm + nt*sn + kb*sk] (128-granular tiles)
    int64_t sm, sn, sk, nt_limit;
    float* C;
    int64_t ldc;
    int32_t* dump;
    const float* s_row;          // dX: 1/s_x[row] rescale
    const float* s_col;          // dW: 1/s_w[col] rescale
    int ec_mode;
    int64_t S, B;
    const float* eps;
    const int32_t* rowsum;
    const float* v;
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

// 10 warps: one SM sub-partition hosts three of them, so 16384 / (3 * 32) caps
// the kernel at 168 registers per thread.
template <int EPI, bool MN>
__global__ void __launch_bounds__(THREADS, 1)
    umma_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, Args P) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ int abort_flag;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_STAGE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * B_STAGE);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
    const uint32_t full0 = su32(bars), empty0 = su32(bars + STAGES), tfull0 = su32(bars + 2 * STAGES),
                   tempty0 = su32(bars + 2 * STAGES + 2), done_bar = su32(bars + 2 * STAGES + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
    const int nkb = (int)s3r_cdiv(P.K, 128);
    const int nslices = 2 * nkb;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8 * b, 1);
            mbar_init(tempty0 + 8 * b, 8);
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

    if (warp == 0) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmA) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmB) : "memory");
            int issued = 0;
            for (int it = 0; it < nslices; ++it) {
                const int s = it % STAGES;
                const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
                if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, abrt)) {
                    *abrt = 1;
                    break;
                }
                const uint32_t fb = full0 + 8 * s;
                mbar_expect_tx(fb, STAGE_BYTES);
                const int32_t k0 = it * BKS;
                const uint32_t a_dst = su32(sA + s * A_STAGE), b_dst = su32(sB + s * B_STAGE);
                if (!MN) {
                    tma_load(a_dst, &tmA, k0, (int32_t)m0, fb);
                    tma_load(b_dst, &tmB, k0, (int32_t)n0, fb);
                } else {
                    tma_load(a_dst, &tmA, (int32_t)m0, k0, fb);
                    tma_load(a_dst + MN_ATOM_BYTES, &tmA, (int32_t)m0 + 64, k0, fb);
#pragma unroll
                    for (int j = 0; j < 4; ++j) tma_load(b_dst + j * MN_ATOM_BYTES, &tmB, (int32_t)n0 + 64 * j, k0, fb);
                }
                issued = it + 1;
            }
            // no copy may still be landing in shared memory when the CTA exits
            for (int it = issued > STAGES ? issued - STAGES : 0; it < issued; ++it)
                mbar_wait(full0 + 8 * (it % STAGES), (uint32_t)(it / STAGES) & 1u, abrt);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(BM, BN, MN, MN);
            for (int kb = 0; kb < nkb; ++kb) {
                const int buf = kb & 1;
                if (!mbar_wait(tempty0 + 8 * buf, ((uint32_t)(kb >> 1) & 1u) ^ 1u, abrt)) {
                    *abrt = 1;
                    break;
                }
                tc_after();
                const uint32_t d_tmem = tmem + (uint32_t)(buf * BN);
                bool ok = true;
                for (int h = 0; h < 2; ++h) {
                    const int it = 2 * kb + h, s = it % STAGES;
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
                if (!ok) {
                    *abrt = 1;
                    break;
                }
                umma_commit(tfull0 + 8 * buf);
            }
            umma_commit(done_bar);
            mbar_wait(done_bar, 0, abrt);
        }
    } else {
        // ------------------------------ epilogue ------------------------------
        const int q = warp & 3, half = (warp - 2) >> 2, ew = warp - 2;
        const int64_t row = m0 + 32 * q + lane;
        const int64_t c0 = n0 + 128 * half;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(128 * half);
        float acc[128];
#pragma unroll
        for (int j = 0; j < 128; ++j) acc[j] = 0.0f;
        const int64_t mt = m0 / 128, nt = n0 / 128 + half;
        const bool has_scale = EPI != kDump && nt < P.nt_limit;
        const float* scale_ptr = has_scale ? P.scale + mt * P.sm + nt * P.sn : nullptr;
        float sc_next = (has_scale && nkb > 0) ? __ldg(scale_ptr) : 0.0f;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
            const int buf = kb & 1;
            const float sc = sc_next;   // loaded one block ahead
            if (has_scale && kb + 1 < nkb) sc_next = __ldg(scale_ptr + (int64_t)(kb + 1) * P.sk);
            // warp-uniform outcome: the tcgen05.ld below needs the whole warp
            const bool got = __all_sync(0xFFFFFFFFu, mbar_wait(tfull0 + 8 * buf, (uint32_t)(kb >> 1) & 1u, abrt));
            if (!got) {
                ok = false;
                *abrt = 1;
                break;
            }
            tc_after();
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint32_t r[16];
                tmem_ld16(lane_addr + (uint32_t)(buf * BN + 16 * c), r);
                tmem_wait_ld();
                if (EPI == kDump) {
                    if (row < P.M) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int64_t col = c0 + 16 * c + j;
                            if (col < P.N)
                                P.dump[(row * P.N + col) * nkb + kb] = __float2int_rn(__uint_as_float(r[j]));
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) acc[16 * c + j] = fmaf(sc, __uint_as_float(r[j]), acc[16 * c + j]);
                }
            }
            tc_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty0 + 8 * buf);
        }
        if (EPI != kDump && ok) {
            // The last accumulator commit retired every MMA, so the operand ring is
            // free: stage this warp's 32 x 128 fp32 block there (row pitch 132
            // floats keeps both the row writes and the column reads conflict-free),
            // then finish row by row with 16-byte coalesced accesses.
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            float* stage = reinterpret_cast<float*>(smem) + ew * (32 * 132);
            float* mine = stage + lane * 132;
#pragma unroll
            for (int c = 0; c < 32; ++c)
                *reinterpret_cast<float4*>(mine + 4 * c) =
                    make_float4(acc[4 * c], acc[4 * c + 1], acc[4 * c + 2], acc[4 * c + 3]);
            __syncwarp();
            const int64_t col = c0 + 4 * lane;   // this thread's 4 columns
            const bool vec = (P.ldc % 4 == 0) && ((reinterpret_cast<uintptr_t>(P.C) & 15u) == 0) && col + 4 <= P.N;
            float cterm[4] = {0.f, 0.f, 0.f, 0.f}, cscale[4] = {1.f, 1.f, 1.f, 1.f};
            if (EPI == kDX) {
                // every row of this tile lies in one example (S % 128 == 0 or one example)
                if (P.ec_mode) {
                    const int64_t b = m0 / P.S;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (col + j < P.N) {
                            cterm[j] = __ldg(P.v + b * P.N + col + j);   // v[b, col]
                            cscale[j] = (float)__ldg(P.rowsum + col + j);
                        }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (col + j < P.N && P.s_col) cscale[j] = __ldg(P.s_col + col + j);
            }
            for (int r = 0; r < 32; ++r) {
                const int64_t grow = m0 + 32 * q + r;
                if (grow >= P.M) break;
                const float4 a4 = *reinterpret_cast<const float4*>(stage + r * 132 + 4 * lane);
                float o[4] = {a4.x, a4.y, a4.z, a4.w};
                float* dst = P.C + grow * P.ldc + col;
                if (EPI == kDX) {
                    const float ep = P.ec_mode ? __ldg(P.eps + grow) : 0.0f;
                    const float sr = P.s_row ? __ldg(P.s_row + grow) : 1.0f;
                    float old[4] = {0.f, 0.f, 0.f, 0.f};
                    if (P.accumulate) {
                        if (vec) {
                            const float4 t = *reinterpret_cast<const float4*>(dst);
                            old[0] = t.x; old[1] = t.y; old[2] = t.z; old[3] = t.w;
                        } else {
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                if (col + j < P.N) old[j] = dst[j];
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (P.ec_mode) o[j] = o[j] - fmaf(ep, cscale[j], cterm[j]);
                        if (P.s_row) o[j] = o[j] / sr;
                        if (P.accumulate) o[j] = o[j] + old[j];
                    }
                } else {
                    if (P.ec_mode == S3R_EC_TWO_WAY) {
                        float corr[4];
                        const float pr = __ldg(P.p + grow);
#pragma unroll
                        for (int j = 0; j < 4; ++j) corr[j] = pr;
                        for (int64_t b = 0; b < P.B; ++b) {
                            const float xs = (float)__ldg(P.xsum + b * P.M + grow);
                            const float m = __ldg(P.mu + b);
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                if (col + j < P.N) corr[j] = fmaf(xs, __ldg(P.colmean + b * P.N + col + j) - m, corr[j]);
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j) o[j] = o[j] - corr[j];
                    }
                    if (P.s_col) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) o[j] = o[j] / cscale[j];
                    }
                }
                if (vec) {
                    *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (col + j < P.N) dst[j] = o[j];
                }
            }
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

template <int EPI, bool MN>
static int launch(const CUtensorMap& a, const CUtensorMap& b, const Args& P, cudaStream_t stream) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e =
            cudaFuncSetAttribute(umma_gemm_kernel<EPI, MN>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return s3r_cuda_fail("umma gemm: cudaFuncSetAttribute", e);
        }
        attr = true;
    }
    if (s3r_cdiv(P.M, BM) > 65535) return S3R_ERR_UNSUPPORTED;
    dim3 grid((unsigned)s3r_cdiv(P.N, BN), (unsigned)s3r_cdiv(P.M, BM));
    umma_gemm_kernel<EPI, MN><<<grid, THREADS, SMEM_BYTES, stream>>>(a, b, P);
    S3R_CHECK_LAUNCH();
    return S3R_OK;
}

}  // namespace umma
}  // namespace s3r

using namespace s3r;

// dX [T, K] from fp16-carried codes: A = Q [T, N], B = W [K, N] (both K-major).
int umma_gemm_dx(const void* Q, const float* tile_scale, const void* W, int64_t T, int64_t N, int64_t K,
                 const float* s_x, int ec_mode, const float* eps, const int32_t* rowsum, const float* v, int64_t S,
                 float* dX, int accumulate, int32_t* dump, int* d_status, cudaStream_t stream) {
    if (!s3r_aligned16(Q) || !s3r_aligned16(W) || N % 8 != 0) return S3R_ERR_ALIGN;
    CUtensorMap ma, mb;
    int st = umma::make_map(&ma, Q, N, T, N, umma::BM);
    if (st) return st;
    st = umma::make_map(&mb, W, N, K, N, umma::BN);
    if (st) return st;
    umma::Args P{};
    P.M = T; P.N = K; P.K = N;
    P.scale = tile_scale; P.sm = s3r_cdiv(N, kTile); P.sn = 0; P.sk = 1; P.nt_limit = INT64_MAX;
    P.C = dX; P.ldc = K; P.dump = dump; P.s_row = s_x; P.ec_mode = ec_mode; P.S = S > 0 ? S : T;
    P.eps = eps; P.rowsum = rowsum; P.v = v; P.accumulate = accumulate; P.d_status = d_status;
    if (dump) return umma::launch<umma::kDump, false>(ma, mb, P, stream);
    return umma::launch<umma::kDX, false>(ma, mb, P, stream);
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
    P.M = K; P.N = N; P.K = T;
    P.scale = tile_scale; P.sm = 0; P.sn = 1; P.sk = s3r_cdiv(N, kTile); P.nt_limit = s3r_cdiv(N, kTile);
    P.C = dW; P.ldc = N; P.dump = dump; P.s_col = s_w; P.ec_mode = ec_mode; P.S = S > 0 ? S : T;
    P.B = S > 0 ? T / S : 1; P.colmean = colmean; P.mu = mu; P.xsum = xsum; P.p = p; P.d_status = d_status;
    if (dump) return umma::launch<umma::kDump, true>(ma, mb, P, stream);
    return umma::launch<umma::kDW, true>(ma, mb, P, stream);
}
