// ffn.cu -- SwiGLU FFN block backward built from the library's entry points,
// and the status helpers.
//
// Paper: "Efficient Quantization Training with Stochastic Rounding via
// Structured Subspace Randomness" §IV-A (single-block SwiGLU FFN benchmark,
// Table III shapes), §III-A..§III-D for each linear.  One stream, no host
// synchronization; every intermediate lives in the caller's workspace.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <set>
#include <utility>
#include <vector>

#include "common.cuh"

#include <cstdio>

static std::atomic<uint64_t> g_launches{0};
void s3r_count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
extern "C" uint64_t s3r_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

static thread_local char g_last_error[512] = "";
void s3r_record_error(const char* where, const char* what) {
    std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s", where, what);
}
int s3r_cuda_fail(const char* where, cudaError_t err) {
    char buf[400];
    std::snprintf(buf, sizeof(buf), "%s (%s)", cudaGetErrorName(err), cudaGetErrorString(err));
    s3r_record_error(where, buf);
    return S3R_ERR_CUDA;
}
extern "C" const char* s3r_last_error(void) { return g_last_error; }

extern "C" int s3r_debug_wait_timeout(int family, uint64_t limit_ns, int raise_abort, int* d_status,
                                      unsigned long long* d_waited_ns, cudaStream_t stream) {
    if (!d_status || !d_waited_ns || limit_ns == 0 || limit_ns > 2000000000ull) return S3R_ERR_ARG;
    switch (family) {
        case S3R_WAIT_GEMM: return umma_wait_probe(limit_ns, raise_abort, d_status, d_waited_ns, stream);
        case S3R_WAIT_QUANTIZE:
            if (raise_abort) return S3R_ERR_ARG;   // the quantizers' waits have no abort flag
            return quant_wait_probe(limit_ns, d_status, d_waited_ns, stream);
        case S3R_WAIT_EC: return ec_wait_probe(limit_ns, raise_abort, d_status, d_waited_ns, stream);
        default: return S3R_ERR_ARG;
    }
}

static std::mutex g_setup_mutex;

int s3r_sm_count() {
    constexpr int kMaxDev = 64;
    static int counts[kMaxDev] = {};
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        (void)cudaGetLastError();
        return 148;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (dev < kMaxDev && counts[dev]) return counts[dev];
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        return 148;
    }
    if (dev < kMaxDev) counts[dev] = n;
    return n;
}

int s3r_kernel_smem(const void* func, int bytes, const char* what) {
    static std::set<std::pair<const void*, int>> done;   // (kernel, device) pairs already raised
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return s3r_cuda_fail(what, e);
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (done.count({func, dev})) return S3R_OK;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return s3r_cuda_fail(what, e);
    }
    done.insert({func, dev});
    return S3R_OK;
}

namespace {

constexpr uint32_t kRhsOffset = S3R_TID_RHS_OFFSET;
constexpr int MaxGroup = 24;   // problems per multi-problem GEMM launch

struct Carver {
    uintptr_t cur, end;
    bool ok = true;
    Carver(void* base, size_t bytes) : cur((uintptr_t)base), end((uintptr_t)base + bytes) {}
    template <typename T>
    T* take(int64_t count) {
        cur = (cur + 255) & ~(uintptr_t)255;
        T* p = reinterpret_cast<T*>(cur);
        cur += (uintptr_t)(count > 0 ? count : 0) * sizeof(T);
        if (cur > end) ok = false;
        return p;
    }
};

// Buffers of one linear's quantization + correction.
struct LinearWs {
    void* Q;         // codes for dX (and dW unless independent SR)
    float* scale;
    void* Qr;        // independent SR: codes for dW
    float* scale_r;
    float* tok;
    float* col;
    float *eps, *mu, *colmean, *v, *p;
    int32_t *rowsum, *xsum;
};

// Carve (or size, when base == nullptr) the whole FFN workspace.
struct FfnLayout {
    LinearWs w2, w1, w3;
    float* dA;
    void* ec_ws;
    size_t ec_ws_bytes;
    void* dw_ws;
    size_t dw_ws_bytes;
    size_t total;
    bool ok;
};

void carve_linear(Carver& c, LinearWs& L, int64_t T, int64_t N, int64_t K, int64_t S, int round_mode, int fmt) {
    const int64_t ntr = s3r_cdiv(T, S3R_TILE), ntc = s3r_cdiv(N, S3R_TILE), B = T / S;
    const int64_t qbytes = T * N * (fmt == S3R_CODES_F16 ? 2 : 1);
    L.Q = c.take<uint8_t>(qbytes);
    L.scale = c.take<float>(ntr * ntc);
    L.Qr = round_mode == S3R_ROUND_INDEP ? c.take<uint8_t>(qbytes) : nullptr;
    L.scale_r = round_mode == S3R_ROUND_INDEP ? c.take<float>(ntr * ntc) : nullptr;
    L.tok = c.take<float>(T * ntc);
    L.col = c.take<float>(ntr * N);
    L.eps = c.take<float>(T);
    L.mu = c.take<float>(B);
    L.colmean = c.take<float>(B * N);
    L.v = c.take<float>(B * K);
    L.p = c.take<float>(K);
    L.rowsum = c.take<int32_t>(K);
    L.xsum = c.take<int32_t>(B * K);
}

FfnLayout layout(void* base, size_t bytes, int64_t T, int64_t d, int64_t F, int64_t S, int round_mode, int fmt) {
    FfnLayout Lo{};
    Carver c(base, base ? bytes : ~(size_t)0 >> 1);
    carve_linear(c, Lo.w2, T, d, F, S, round_mode, fmt);   // W2: G = dY [T, d], W2 [F, d]
    carve_linear(c, Lo.w1, T, F, d, S, round_mode, fmt);   // W1: G = dh1 [T, F], W1 [d, F]
    carve_linear(c, Lo.w3, T, F, d, S, round_mode, fmt);
    Lo.dA = c.take<float>(T * F);
    {   // W2's factors read A8 [T, F]; W1 and W3 share one pass over X8 [T, d]
        const size_t a = s3r_ec_workspace_size(T, F), b = s3r_ec_pair_workspace_size(T, d);
        Lo.ec_ws_bytes = a > b ? a : b;
    }
    Lo.ec_ws = c.take<uint8_t>((int64_t)Lo.ec_ws_bytes);
    const size_t a = int8_gemm_dw_workspace_size(T, F, d, fmt), b = int8_gemm_dw_workspace_size(T, d, F, fmt);
    Lo.dw_ws_bytes = a > b ? a : b;
    Lo.dw_ws = c.take<uint8_t>((int64_t)Lo.dw_ws_bytes);
    Lo.total = (size_t)(c.cur - (uintptr_t)base) + 256;
    Lo.ok = c.ok;
    return Lo;
}

#define S3R_TRY(expr)             \
    do {                          \
        int _st = (expr);         \
        if (_st != S3R_OK) return _st; \
    } while (0)

}  // namespace

// S3R_CODES_S8_F16: the fp16 copies of the five operand code tensors follow the
// fp16 block's workspace (E experts' stacked weights in grouped mode).
size_t widen_bytes(int64_t T, int64_t d, int64_t F, int64_t E) {
    auto r = [](int64_t b) { return (size_t)((b + 255) / 256 * 256); };
    return 255 + r(2 * T * d) + r(2 * T * F) + 2 * r(2 * E * d * F) + r(2 * E * F * d);
}

// S3R_FFN_RECOMPUTE_A: the recomputed codes of a [T, F] (in the format the block computes in)
// and their scales [T] follow everything else.
size_t recompute_bytes(int64_t T, int64_t F, int fmt) {
    auto r = [](int64_t b) { return (size_t)((b + 255) / 256 * 256); };
    return 255 + r(T * F * (fmt == S3R_CODES_S8 ? 1 : 2)) + r(4 * T);
}

extern "C" size_t s3r_ffn_workspace_size(int64_t T, int64_t d, int64_t F, int64_t S, int round_mode, int ec_mode,
                                         int code_format) {
    (void)ec_mode;
    if (T <= 0 || d <= 0 || F <= 0 || S <= 0 || T % S != 0) return 0;
    if (code_format == S3R_CODES_S8_F16)
        return layout(nullptr, 0, T, d, F, S, round_mode, S3R_CODES_F16).total + widen_bytes(T, d, F, 1);
    return layout(nullptr, 0, T, d, F, S, round_mode, code_format).total;
}

namespace {

// One example group's backward (the whole batch, or one expert's rows):
// the argument view, its workspace carve, tensor ids tid_base + (0, 1, 2).
struct Block {
    s3r_ffn_args a;
    FfnLayout Lo;
    int rm, ec, fmt;
    bool indep;
    uint32_t tid2, tid1, tid3;
    int ec2_ctas = 0, ec13_ctas = 0;   // grid caps of the EC streaming passes (0: all SMs)
};

int make_block(Block& b, const s3r_ffn_args& a, void* ws, size_t ws_bytes, uint32_t tid_base) {
    b.a = a;
    b.fmt = a.code_format;
    b.Lo = layout(ws, ws_bytes, a.T, a.d, a.F, a.S, a.round_mode, b.fmt);
    if (!b.Lo.ok) return S3R_ERR_WORKSPACE;
    b.rm = a.round_mode;
    const bool shared = b.rm == S3R_ROUND_S3R || b.rm == S3R_ROUND_S3R_7BIT || b.rm == S3R_ROUND_BCAST;
    b.ec = shared ? a.ec_mode : S3R_EC_NONE;
    b.indep = b.rm == S3R_ROUND_INDEP;
    b.tid2 = tid_base + S3R_TID_W2;
    b.tid1 = tid_base + S3R_TID_W1;
    b.tid3 = tid_base + S3R_TID_W3;
    return S3R_OK;
}

// 1. quantize dY with the W2 fold (s_a per token, s_w2 per output channel)
int step_quantize_dy(Block& b, cudaStream_t stream) {
    const s3r_ffn_args& a = b.a;
    LinearWs& L2 = b.Lo.w2;
    const int64_t T = a.T, d = a.d;
    if (b.rm == S3R_ROUND_S3R || b.rm == S3R_ROUND_S3R_7BIT || b.rm == S3R_ROUND_BCAST)
        return s3r_quantize_ex(a.dY, T, d, d, a.s_a, a.s_w2, b.rm, a.S, nullptr, a.seed, b.tid2, L2.Q, b.fmt,
                               L2.scale, L2.tok, L2.col, a.d_status, stream);
    if (b.indep) {
        S3R_TRY(indep_sr_quantize(a.dY, T, d, d, a.s_a, a.s_w2, a.seed, b.tid2, L2.Q, b.fmt, L2.scale, a.d_status,
                                  stream));
        return indep_sr_quantize(a.dY, T, d, d, a.s_a, a.s_w2, a.seed, b.tid2 + kRhsOffset, L2.Qr, b.fmt,
                                 L2.scale_r, a.d_status, stream);
    }
    return rtne_quantize(a.dY, T, d, d, a.s_a, a.s_w2, S3R_AXIS_TILE, L2.Q, b.fmt, L2.scale, a.d_status, stream);
}

// 2. correction factors of W2 (W8 = W2_8 [F, d], X8 = A8 [T, F])
int step_ec_w2(Block& b, cudaStream_t stream) {
    if (b.ec == S3R_EC_NONE) return S3R_OK;
    const s3r_ffn_args& a = b.a;
    LinearWs& L2 = b.Lo.w2;
    return s3r_ec_correct_capped(L2.tok, L2.col, a.T, a.d, a.S, a.W2_8, a.F, a.A8, b.fmt, b.ec, L2.eps, L2.mu,
                                 L2.colmean, L2.rowsum, L2.v, L2.xsum, L2.p, b.Lo.ec_ws, b.Lo.ec_ws_bytes, b.ec2_ctas,
                                 a.d_status, stream);
}

// 3. dA = Q2 W2_8^T (rescaled, corrected, / s_a)  [T, F]
UmmaDxProblem dx_problem_da(const Block& b) {
    const s3r_ffn_args& a = b.a;
    const LinearWs& L2 = b.Lo.w2;
    return UmmaDxProblem{L2.Q, L2.scale, a.W2_8, L2.eps, L2.rowsum, L2.v, nullptr, nullptr, nullptr, nullptr, nullptr,
                         nullptr, a.T, a.d, a.F, a.s_a, b.ec, a.S, b.Lo.dA, 0, nullptr};
}
int step_da(Block& b, cudaStream_t stream) {
    const s3r_ffn_args& a = b.a;
    const LinearWs& L2 = b.Lo.w2;
    return int8_gemm_dx(L2.Q, L2.scale, a.W2_8, b.fmt, a.T, a.d, a.F, a.s_a, b.ec, L2.eps, L2.rowsum, L2.v, a.S,
                        b.Lo.dA, 0, a.d_status, stream);
}

// 4. dW2 = A8^T Q2 / s_w2  [F, d]
UmmaDwProblem dw_problem(const Block& b, const void* X8, const LinearWs& L, int64_t K, int64_t N, const float* s_w,
                         float* dW) {
    const bool two = b.ec == S3R_EC_TWO_WAY || b.ec == S3R_EC_DW_ONLY;
    return UmmaDwProblem{X8, b.indep ? L.Qr : L.Q, b.indep ? L.scale_r : L.scale, b.a.T, K, N, s_w, b.ec,
                         two ? L.colmean : nullptr, two ? L.mu : nullptr, two ? L.xsum : nullptr,
                         two ? L.p : nullptr, b.a.S, dW, nullptr};
}
int step_dw2(Block& b, cudaStream_t stream) {
    const s3r_ffn_args& a = b.a;
    const LinearWs& L2 = b.Lo.w2;
    return int8_gemm_dw(a.A8, b.indep ? L2.Qr : L2.Q, b.indep ? L2.scale_r : L2.scale, b.fmt, a.T, a.F, a.d, a.s_w2,
                        b.ec, L2.colmean, L2.mu, L2.xsum, L2.p, a.S, a.dW2, b.Lo.dw_ws, b.Lo.dw_ws_bytes, a.d_status,
                        stream);
}

// 5. SwiGLU glue fused into the quantization of dh1 (W1 fold) and dh3 (W3 fold)
int step_swiglu(Block& b, cudaStream_t stream) {
    const s3r_ffn_args& a = b.a;
    LinearWs &L1 = b.Lo.w1, &L3 = b.Lo.w3;
    const int64_t T = a.T, F = a.F;
    const bool keep_err = b.ec != S3R_EC_NONE;
    S3R_TRY(swiglu_quantize_ex(b.Lo.dA, F, a.h1, a.h3, F, T, F, a.s_x, a.s_w1, a.s_w3, b.rm, a.S, b.fmt, a.seed, b.tid1,
                            b.tid3, L1.Q, L1.scale, keep_err ? L1.tok : nullptr, keep_err ? L1.col : nullptr, L3.Q,
                            L3.scale, keep_err ? L3.tok : nullptr, keep_err ? L3.col : nullptr, a.d_status, stream));
    if (b.indep)
        S3R_TRY(swiglu_quantize_ex(b.Lo.dA, F, a.h1, a.h3, F, T, F, a.s_x, a.s_w1, a.s_w3, b.rm, a.S, b.fmt, a.seed,
                                b.tid1 + kRhsOffset, b.tid3 + kRhsOffset, L1.Qr, L1.scale_r, nullptr, nullptr, L3.Qr,
                                L3.scale_r, nullptr, nullptr, a.d_status, stream));
    return S3R_OK;
}

// 3 + 4 + 5 with the glue in the dA epilogue (fp16 codes; not independent SR):
// the glue's description for the dA problem of the mixed launch
UmmaGlue glue_of(const Block& b) {
    const s3r_ffn_args& a = b.a;
    const LinearWs &L1 = b.Lo.w1, &L3 = b.Lo.w3;
    const bool keep_err = b.ec != S3R_EC_NONE;
    UmmaGlue g{};
    g.dx_index = 0;
    g.round_mode = b.rm;
    g.seed = a.seed;
    g.tid1 = b.tid1;
    g.tid3 = b.tid3;
    g.S = a.S;
    g.h1 = a.h1;
    g.h3 = a.h3;
    g.ldh = a.F;
    g.s_x = a.s_x;
    g.s_w1 = a.s_w1;
    g.s_w3 = a.s_w3;
    g.Q1 = L1.Q;
    g.Q3 = L3.Q;
    g.scale1 = L1.scale;
    g.scale3 = L3.scale;
    g.tok1 = keep_err ? L1.tok : nullptr;
    g.tok3 = keep_err ? L3.tok : nullptr;
    g.col1 = keep_err ? L1.col : nullptr;
    g.col3 = keep_err ? L3.col : nullptr;
    return g;
}

// 6. correction factors of W1 and W3 (W8 [d, F], X8 [T, d]), one pass over X8
int step_ec_w13(Block& b, cudaStream_t stream) {
    if (b.ec == S3R_EC_NONE) return S3R_OK;
    const s3r_ffn_args& a = b.a;
    LinearWs &L1 = b.Lo.w1, &L3 = b.Lo.w3;
    return s3r_ec_correct_pair(L1.tok, L1.col, a.W1_8, L1.eps, L1.mu, L1.colmean, L1.rowsum, L1.v, L1.xsum, L1.p,
                               L3.tok, L3.col, a.W3_8, L3.eps, L3.mu, L3.colmean, L3.rowsum, L3.v, L3.xsum, L3.p,
                               a.T, a.F, a.S, a.d, a.X8, b.fmt, b.ec, b.Lo.ec_ws, b.Lo.ec_ws_bytes, b.ec13_ctas,
                               a.d_status, stream);
}

// 7. dX = dX1 + dX3
UmmaDxProblem dx_problem_dx(const Block& b) {
    const s3r_ffn_args& a = b.a;
    const LinearWs &L1 = b.Lo.w1, &L3 = b.Lo.w3;
    return UmmaDxProblem{L1.Q, L1.scale, a.W1_8, L1.eps, L1.rowsum, L1.v, L3.Q, L3.scale, a.W3_8, L3.eps, L3.rowsum,
                         L3.v, a.T, a.F, a.d, a.s_x, b.ec, a.S, a.dX, 0, nullptr};
}
int step_dx(Block& b, cudaStream_t stream) {
    const s3r_ffn_args& a = b.a;
    const LinearWs &L1 = b.Lo.w1, &L3 = b.Lo.w3;
    const s3r_dx_term terms[2] = {{L1.Q, L1.scale, a.W1_8, L1.eps, L1.rowsum, L1.v},
                                  {L3.Q, L3.scale, a.W3_8, L3.eps, L3.rowsum, L3.v}};
    return int8_gemm_dx_sum(terms, 2, b.fmt, a.T, a.F, a.d, a.s_x, b.ec, a.S, a.dX, 0, a.d_status, stream);
}

// 8. dW1, dW3 (fp16 codes: both in one persistent launch, their tiles share the grid)
int step_dw13(Block& b, cudaStream_t stream) {
    const s3r_ffn_args& a = b.a;
    const LinearWs &L1 = b.Lo.w1, &L3 = b.Lo.w3;
    if (b.fmt == S3R_CODES_F16) {
        const UmmaDwProblem q[2] = {dw_problem(b, a.X8, L1, a.d, a.F, a.s_w1, a.dW1),
                                    dw_problem(b, a.X8, L3, a.d, a.F, a.s_w3, a.dW3)};
        return umma_dw_group(q, 2, a.d_status, stream);
    }
    S3R_TRY(int8_gemm_dw(a.X8, b.indep ? L1.Qr : L1.Q, b.indep ? L1.scale_r : L1.scale, b.fmt, a.T, a.d, a.F, a.s_w1,
                         b.ec, L1.colmean, L1.mu, L1.xsum, L1.p, a.S, a.dW1, b.Lo.dw_ws, b.Lo.dw_ws_bytes,
                         a.d_status, stream));
    return int8_gemm_dw(a.X8, b.indep ? L3.Qr : L3.Q, b.indep ? L3.scale_r : L3.scale, b.fmt, a.T, a.d, a.F, a.s_w3,
                        b.ec, L3.colmean, L3.mu, L3.xsum, L3.p, a.S, a.dW3, b.Lo.dw_ws, b.Lo.dw_ws_bytes, a.d_status,
                        stream);
}

int record(const s3r_ffn_args* a, int i, cudaStream_t stream) {
    if (!a->step_events) return S3R_OK;
    cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(a->step_events[i]), stream);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return s3r_cuda_fail("ffn_backward step event", e);
    }
    return S3R_OK;
}

// Rows of expert e in grouped mode: the argument view with every per-row
// pointer moved to the group's first row and every per-expert pointer to
// the expert's slice.
s3r_ffn_args expert_view(const s3r_ffn_args& a, int64_t e, int64_t r0, int64_t Tg) {
    const int64_t d = a.d, F = a.F;
    const size_t cs = a.code_format == S3R_CODES_F16 ? 2 : 1;
    s3r_ffn_args g = a;
    g.T = Tg;
    g.S = Tg;
    g.num_groups = 0;
    g.group_offsets = nullptr;
    g.dY = static_cast<const uint16_t*>(a.dY) + r0 * d;
    g.h1 = static_cast<const uint16_t*>(a.h1) + r0 * F;
    g.h3 = static_cast<const uint16_t*>(a.h3) + r0 * F;
    g.X8 = static_cast<const uint8_t*>(a.X8) + (size_t)(r0 * d) * cs;
    g.s_x = a.s_x ? a.s_x + r0 : nullptr;
    g.A8 = static_cast<const uint8_t*>(a.A8) + (size_t)(r0 * F) * cs;
    g.s_a = a.s_a ? a.s_a + r0 : nullptr;
    g.W1_8 = static_cast<const uint8_t*>(a.W1_8) + (size_t)(e * d * F) * cs;
    g.s_w1 = a.s_w1 ? a.s_w1 + e * F : nullptr;
    g.W3_8 = static_cast<const uint8_t*>(a.W3_8) + (size_t)(e * d * F) * cs;
    g.s_w3 = a.s_w3 ? a.s_w3 + e * F : nullptr;
    g.W2_8 = static_cast<const uint8_t*>(a.W2_8) + (size_t)(e * F * d) * cs;
    g.s_w2 = a.s_w2 ? a.s_w2 + e * d : nullptr;
    g.dX = a.dX + r0 * d;
    g.dW1 = a.dW1 + e * d * F;
    g.dW3 = a.dW3 + e * d * F;
    g.dW2 = a.dW2 + e * F * d;
    return g;
}

// Side streams for the grouped mode's per-expert memory-bound steps (EC,
// quantize, SwiGLU): expert e's launches of such a step go to side stream
// e % kSideStreams, forked from and joined back to the caller's stream with
// events, so small experts' kernels overlap instead of running one after
// another.  Created once per device (non-blocking streams and timing-free
// events); the fork and join are plain event waits, so a stream capture of
// the caller's stream captures them as graph edges.  The pool is per host
// thread (two threads' calls never share its events) and lives until exit.
constexpr int kSideStreams = 4;
struct SidePool {
    cudaStream_t s[kSideStreams];
    cudaEvent_t fork, join[kSideStreams];
    bool ok = false;
};
thread_local SidePool g_side[64];

int side_pool(SidePool** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return s3r_cuda_fail("ffn_backward: cudaGetDevice", e == cudaSuccess ? cudaErrorInvalidDevice : e);
    }
    SidePool& p = g_side[dev];
    if (!p.ok) {
        for (int i = 0; i < kSideStreams && e == cudaSuccess; ++i)
            e = cudaStreamCreateWithFlags(&p.s[i], cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.fork, cudaEventDisableTiming);
        for (int i = 0; i < kSideStreams && e == cudaSuccess; ++i)
            e = cudaEventCreateWithFlags(&p.join[i], cudaEventDisableTiming);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return s3r_cuda_fail("ffn_backward: side streams", e);
        }
        p.ok = true;
    }
    *out = &p;
    return S3R_OK;
}

// Runs step(b, stream) for every block, block i on side stream i % kSideStreams,
// between a fork from and a join back to `main`.
template <typename Step>
int run_on_side_streams(std::vector<Block>& blocks, Step step, cudaStream_t main) {
    SidePool* p = nullptr;
    S3R_TRY(side_pool(&p));
    const int used = (int)std::min<size_t>(blocks.size(), (size_t)kSideStreams);
    cudaError_t e = cudaEventRecord(p->fork, main);
    for (int i = 0; i < used && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(p->s[i], p->fork, 0);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return s3r_cuda_fail("ffn_backward: fork", e);
    }
    int st = S3R_OK;
    for (size_t i = 0; i < blocks.size() && st == S3R_OK; ++i) st = step(blocks[i], p->s[i % kSideStreams]);
    // join every side stream that was forked, also after a failure
    for (int i = 0; i < used && e == cudaSuccess; ++i) {
        e = cudaEventRecord(p->join[i], p->s[i]);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(main, p->join[i], 0);
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return s3r_cuda_fail("ffn_backward: join", e);
    }
    return st;
}

// Workspace of the grouped mode: one block carve per non-empty expert, side by side.
size_t grouped_bytes(const int64_t* off, int64_t E, int64_t d, int64_t F, int round_mode, int fmt) {
    size_t total = 0;
    for (int64_t e = 0; e < E; ++e) {
        const int64_t Tg = off[e + 1] - off[e];
        if (Tg > 0) total += layout(nullptr, 0, Tg, d, F, Tg, round_mode, fmt).total + 256;
    }
    return total;
}

}  // namespace

extern "C" size_t s3r_ffn_workspace_size_flags(int64_t T, int64_t d, int64_t F, int64_t S, int round_mode,
                                               int ec_mode, int code_format, int flags) {
    const size_t n = s3r_ffn_workspace_size(T, d, F, S, round_mode, ec_mode, code_format);
    return n && (flags & S3R_FFN_RECOMPUTE_A) ? n + recompute_bytes(T, F, code_format) : n;
}

extern "C" size_t s3r_ffn_grouped_workspace_size(const int64_t* group_offsets, int64_t num_groups, int64_t d,
                                                 int64_t F, int round_mode, int ec_mode, int code_format) {
    (void)ec_mode;
    if (!group_offsets || num_groups <= 0 || d <= 0 || F <= 0) return 0;
    for (int64_t e = 0; e < num_groups; ++e)
        if (group_offsets[e + 1] < group_offsets[e]) return 0;
    if (code_format == S3R_CODES_S8_F16)
        return grouped_bytes(group_offsets, num_groups, d, F, round_mode, S3R_CODES_F16) +
               widen_bytes(group_offsets[num_groups] - group_offsets[0], d, F, num_groups);
    return grouped_bytes(group_offsets, num_groups, d, F, round_mode, code_format);
}

extern "C" size_t s3r_ffn_grouped_workspace_size_flags(const int64_t* group_offsets, int64_t num_groups, int64_t d,
                                                       int64_t F, int round_mode, int ec_mode, int code_format,
                                                       int flags) {
    const size_t n = s3r_ffn_grouped_workspace_size(group_offsets, num_groups, d, F, round_mode, ec_mode, code_format);
    if (!n || !(flags & S3R_FFN_RECOMPUTE_A)) return n;
    return n + recompute_bytes(group_offsets[num_groups] - group_offsets[0], F, code_format);
}

extern "C" int s3r_ffn_workspace_offsets(int64_t T, int64_t d, int64_t F, int64_t S, int round_mode,
                                         int code_format, const int64_t* group_offsets, int64_t num_groups,
                                         int64_t group, size_t* out) {
    if (!out || d <= 0 || F <= 0) return S3R_ERR_ARG;
    if (code_format == S3R_CODES_S8_F16) code_format = S3R_CODES_F16;   // the widened block runs on fp16 codes
    if (code_format != S3R_CODES_S8 && code_format != S3R_CODES_F16) return S3R_ERR_ARG;
    uintptr_t base = 0;   // offsets from a 256-byte aligned workspace base
    if (num_groups > 0) {
        if (!group_offsets || group < 0 || group >= num_groups || group_offsets[0] != 0) return S3R_ERR_ARG;
        for (int64_t e = 0; e < num_groups; ++e)
            if (group_offsets[e + 1] < group_offsets[e]) return S3R_ERR_ARG;
        // the same walk as ffn_backward's grouped carve: one block per non-empty expert
        for (int64_t e = 0; e < group; ++e) {
            const int64_t Tg = group_offsets[e + 1] - group_offsets[e];
            if (Tg == 0) continue;
            base = (base + 255) & ~(uintptr_t)255;
            base += layout(nullptr, 0, Tg, d, F, Tg, round_mode, code_format).total;
        }
        base = (base + 255) & ~(uintptr_t)255;
        T = group_offsets[group + 1] - group_offsets[group];
        S = T;
    }
    if (T <= 0 || S <= 0 || T % S != 0) return S3R_ERR_ARG;
    const FfnLayout Lo = layout(nullptr, 0, T, d, F, S, round_mode, code_format);
    const void* views[S3R_FFN_WS_VIEWS] = {Lo.w2.Q, Lo.w2.scale, Lo.w1.Q, Lo.w1.scale, Lo.w3.Q, Lo.w3.scale, Lo.dA};
    for (int i = 0; i < S3R_FFN_WS_VIEWS; ++i) out[i] = (size_t)(base + reinterpret_cast<uintptr_t>(views[i]));
    return S3R_OK;
}

namespace {

// The host checks of ffn_backward that need no workspace carve: sizes, modes,
// pointers, the example split (dense) or the row offsets (grouped).
int check_block_args(const s3r_ffn_args* a) {
    if (!a) return S3R_ERR_ARG;
    const int64_t T = a->T, d = a->d, F = a->F, S = a->S;
    if (T <= 0 || d <= 0 || F <= 0) return S3R_ERR_ARG;
    if (a->round_mode < S3R_ROUND_RTNE || a->round_mode > S3R_ROUND_BCAST) return S3R_ERR_ARG;
    if (a->ec_mode < S3R_EC_NONE || a->ec_mode > S3R_EC_DW_ONLY) return S3R_ERR_ARG;
    if (a->code_format != S3R_CODES_S8 && a->code_format != S3R_CODES_F16 && a->code_format != S3R_CODES_S8_F16)
        return S3R_ERR_ARG;
    if (!a->dY || !a->h1 || !a->h3 || !a->X8 || !a->W1_8 || !a->W3_8 || !a->W2_8 || !a->dX || !a->dW1 || !a->dW2 ||
        !a->dW3)
        return S3R_ERR_ARG;
    // A8 and s_a come from the caller, or (S3R_FFN_RECOMPUTE_A) from the call itself
    if ((a->flags & S3R_FFN_RECOMPUTE_A) ? (a->A8 || a->s_a) : !a->A8) return S3R_ERR_ARG;
    if (a->num_groups == 0) {
        if (S <= 0) return S3R_ERR_ARG;
        if (T % S != 0 || (S % S3R_TILE != 0 && S != T)) return S3R_ERR_SHAPE;
        return S3R_OK;
    }
    const int64_t E = a->num_groups;
    const int64_t* off = a->group_offsets;
    if (E < 0 || !off || off[0] != 0 || off[E] != T) return S3R_ERR_ARG;
    for (int64_t e = 0; e < E; ++e)
        if (off[e + 1] < off[e]) return S3R_ERR_ARG;
    if (E > (int64_t)(0xFFFFFFFFu / S3R_MOE_TID_STRIDE)) return S3R_ERR_ARG;
    return S3R_OK;
}

// int8 codes to the same integers in fp16, four at a time: the bytes, offset
// by 128, become the low mantissa bits of 0x6400 (1024 + u exactly), and one
// subtraction of 1152 leaves u - 128, the code, without rounding.
__device__ __forceinline__ void widen4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(0x64646464u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}

struct WidenJob {
    const int8_t* src;
    uint16_t* dst;   // 16-byte aligned
    int64_t n;
};
struct WidenJobs {
    WidenJob j[5];
    int n;
};

__global__ void __launch_bounds__(256) widen_codes_kernel(const WidenJobs J) {
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x, nth = (int64_t)gridDim.x * blockDim.x;
    for (int s = 0; s < J.n; ++s) {
        const WidenJob w = J.j[s];
        const int64_t n16 = ((uintptr_t)w.src & 15u) == 0 ? w.n / 16 : 0;
        const uint4* src = reinterpret_cast<const uint4*>(w.src);
        uint4* dst = reinterpret_cast<uint4*>(w.dst);
        for (int64_t i = tid; i < n16; i += nth) {
            const uint4 v = __ldcs(src + i);
            uint4 a, b;
            widen4(v.x, a.x, a.y);
            widen4(v.y, a.z, a.w);
            widen4(v.z, b.x, b.y);
            widen4(v.w, b.z, b.w);
            dst[2 * i] = a;
            dst[2 * i + 1] = b;
        }
        for (int64_t i = n16 * 16 + tid; i < w.n; i += nth) {
            uint32_t lo, hi;
            widen4((uint32_t)(uint8_t)w.src[i], lo, hi);
            w.dst[i] = (uint16_t)(lo & 0xFFFFu);
        }
    }
}

// S3R_CODES_S8_F16: widens X8, A8, W1_8, W3_8 and W2_8 into the tail of the
// workspace, then runs the fp16-code block on the copies.
int ffn_backward_widened(const s3r_ffn_args* a, cudaStream_t stream, const void* A8_f16 = nullptr) {
    const int64_t T = a->T, d = a->d, F = a->F;   // the arguments passed check_block_args
    const bool grouped = a->num_groups > 0;
    const int64_t E = grouped ? a->num_groups : 1;
    if (d % 8 != 0 || F % 8 != 0) return S3R_ERR_ALIGN;   // the fp16-code GEMMs' rows
    const size_t base = grouped ? s3r_ffn_grouped_workspace_size(a->group_offsets, E, d, F, a->round_mode,
                                                                  a->ec_mode, S3R_CODES_F16)
                                : s3r_ffn_workspace_size(T, d, F, a->S, a->round_mode, a->ec_mode, S3R_CODES_F16);
    if (base == 0) return S3R_ERR_ARG;
    if (!a->workspace || a->workspace_bytes < base + widen_bytes(T, d, F, E)) return S3R_ERR_WORKSPACE;
    s3r_ffn_args w = *a;
    w.code_format = S3R_CODES_F16;
    w.workspace_bytes = base;
    uintptr_t p = ((uintptr_t)a->workspace + base + 255) & ~(uintptr_t)255;
    WidenJobs J{};
    const void* src[5] = {a->X8, a->A8, a->W1_8, a->W3_8, a->W2_8};
    const int64_t n[5] = {T * d, T * F, E * d * F, E * d * F, E * F * d};
    const void** dst[5] = {&w.X8, &w.A8, &w.W1_8, &w.W3_8, &w.W2_8};
    J.n = 0;
    for (int i = 0; i < 5; ++i) {
        if (i == 1 && A8_f16) {   // the codes of a are fp16 already (recomputed by the call)
            w.A8 = A8_f16;
        } else {
            J.j[J.n++] = WidenJob{static_cast<const int8_t*>(src[i]), reinterpret_cast<uint16_t*>(p), n[i]};
            *dst[i] = reinterpret_cast<const void*>(p);
        }
        p += (uintptr_t)((2 * n[i] + 255) / 256 * 256);
    }
    int64_t total16 = 0;
    for (int i = 0; i < J.n; ++i) total16 += J.j[i].n / 16;
    const int64_t cap = (int64_t)s3r_sm_count() * 8;
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(cap, (total16 + 255) / 256));
    widen_codes_kernel<<<grid, 256, 0, stream>>>(J);
    S3R_CHECK_LAUNCH();
    return ffn_backward(&w, stream);
}

// S3R_FFN_RECOMPUTE_A: the codes of a and their scales from h1 and h3 with the
// forward's own kernel (swiglu_fwd_quantize: a = bf16(silu(h1) h3), per-token
// RTNE), into the tail of the workspace, then the block on them.
int ffn_backward_recompute(const s3r_ffn_args* a, cudaStream_t stream) {
    const int64_t T = a->T, d = a->d, F = a->F;   // the arguments passed check_block_args
    const int fmt = a->code_format, ifmt = fmt == S3R_CODES_S8 ? S3R_CODES_S8 : S3R_CODES_F16;
    const size_t base = a->num_groups > 0
                            ? s3r_ffn_grouped_workspace_size(a->group_offsets, a->num_groups, d, F, a->round_mode,
                                                             a->ec_mode, fmt)
                            : s3r_ffn_workspace_size(T, d, F, a->S, a->round_mode, a->ec_mode, fmt);
    if (base == 0) return S3R_ERR_ARG;
    if (!a->workspace || a->workspace_bytes < base + recompute_bytes(T, F, fmt)) return S3R_ERR_WORKSPACE;
    if (F % 8 != 0 || !s3r_aligned16(a->h1) || !s3r_aligned16(a->h3)) return S3R_ERR_ALIGN;
    uintptr_t p = ((uintptr_t)a->workspace + base + 255) & ~(uintptr_t)255;
    void* A8 = reinterpret_cast<void*>(p);
    p += (uintptr_t)((T * F * (ifmt == S3R_CODES_S8 ? 1 : 2) + 255) / 256 * 256);
    float* s_a = reinterpret_cast<float*>(p);
    S3R_TRY(swiglu_fwd_quantize(a->h1, a->h3, T, F, F, nullptr, A8, ifmt, s_a, a->d_status, stream));
    s3r_ffn_args w = *a;
    w.flags &= ~S3R_FFN_RECOMPUTE_A;
    w.workspace_bytes = base;
    w.s_a = s_a;
    if (fmt == S3R_CODES_S8_F16) return ffn_backward_widened(&w, stream, A8);
    w.A8 = A8;
    return ffn_backward(&w, stream);
}

}  // namespace

extern "C" int ffn_backward(const struct s3r_ffn_args* a, cudaStream_t stream) {
    S3R_TRY(check_block_args(a));
    if (a->flags & S3R_FFN_RECOMPUTE_A) return ffn_backward_recompute(a, stream);
    if (a->code_format == S3R_CODES_S8_F16) return ffn_backward_widened(a, stream);
    const int64_t T = a->T, d = a->d, F = a->F, S = a->S;
    const int fmt = a->code_format;
    if (a->num_groups == 0) {
        if (!a->workspace || a->workspace_bytes < s3r_ffn_workspace_size(T, d, F, S, a->round_mode, a->ec_mode, fmt))
            return S3R_ERR_WORKSPACE;
        Block b;
        S3R_TRY(make_block(b, *a, a->workspace, a->workspace_bytes, 0));
        S3R_TRY(record(a, 0, stream));
        S3R_TRY(step_quantize_dy(b, stream));
        S3R_TRY(record(a, 1, stream));
        S3R_TRY(step_ec_w2(b, stream));
        S3R_TRY(record(a, 2, stream));
        const bool fuse = (a->flags & S3R_FFN_FUSE_GLUE) && fmt == S3R_CODES_F16 && !b.indep;
        if (fuse) {
            // dA (never stored: the SwiGLU glue and the quantization of dh1, dh3 run in its
            // epilogue) and dW2 in one launch; steps 4 and 5 are then empty
            UmmaDxProblem qx = dx_problem_da(b);
            qx.dX = nullptr;
            const UmmaDwProblem qw = dw_problem(b, b.a.A8, b.Lo.w2, b.a.F, b.a.d, b.a.s_w2, b.a.dW2);
            const UmmaGlue gl = glue_of(b);
            S3R_TRY(umma_mixed_group_glue(&qx, 1, &qw, 1, &gl, a->d_status, stream));
            S3R_TRY(record(a, 3, stream));
            S3R_TRY(record(a, 4, stream));
        } else if (fmt == S3R_CODES_F16) {
            // dA and dW2 in one mixed launch (their tiles share the grid); step 4 is then empty
            const UmmaDxProblem qx = dx_problem_da(b);
            const UmmaDwProblem qw = dw_problem(b, b.a.A8, b.Lo.w2, b.a.F, b.a.d, b.a.s_w2, b.a.dW2);
            S3R_TRY(umma_mixed_group(&qx, 1, &qw, 1, a->d_status, stream));
            S3R_TRY(record(a, 3, stream));
            S3R_TRY(record(a, 4, stream));
        } else {
            S3R_TRY(step_da(b, stream));
            S3R_TRY(record(a, 3, stream));
            S3R_TRY(step_dw2(b, stream));
            S3R_TRY(record(a, 4, stream));
        }
        if (!fuse) S3R_TRY(step_swiglu(b, stream));
        S3R_TRY(record(a, 5, stream));
        S3R_TRY(step_ec_w13(b, stream));
        S3R_TRY(record(a, 6, stream));
        if (fmt == S3R_CODES_F16) {
            // dX1 + dX3, dW1 and dW3 in one mixed launch; step 8 is then empty
            const UmmaDxProblem qx = dx_problem_dx(b);
            const UmmaDwProblem qw[2] = {dw_problem(b, b.a.X8, b.Lo.w1, b.a.d, b.a.F, b.a.s_w1, b.a.dW1),
                                         dw_problem(b, b.a.X8, b.Lo.w3, b.a.d, b.a.F, b.a.s_w3, b.a.dW3)};
            S3R_TRY(umma_mixed_group(&qx, 1, qw, 2, a->d_status, stream));
            S3R_TRY(record(a, 7, stream));
        } else {
            S3R_TRY(step_dx(b, stream));
            S3R_TRY(record(a, 7, stream));
            S3R_TRY(step_dw13(b, stream));
        }
        return record(a, 8, stream);
    }
    // grouped: expert e owns rows offsets[e] .. offsets[e+1] (one example);
    // weights, their scales and gradients are stacked per expert.  Every step
    // runs for all experts before the next; with fp16 codes each GEMM step is
    // one multi-problem launch over the experts.
    const int64_t E = a->num_groups;
    const int64_t* off = a->group_offsets;
    if (!a->workspace || a->workspace_bytes < grouped_bytes(off, E, d, F, a->round_mode, fmt))
        return S3R_ERR_WORKSPACE;
    std::vector<Block> blocks;
    blocks.reserve((size_t)E);
    uintptr_t cur = (uintptr_t)a->workspace, end = cur + a->workspace_bytes;
    for (int64_t e = 0; e < E; ++e) {
        const int64_t r0 = off[e], Tg = off[e + 1] - off[e];
        if (Tg == 0) {   // an expert without rows has zero weight gradients
            cudaError_t m = cudaMemsetAsync(a->dW1 + e * d * F, 0, (size_t)(d * F) * sizeof(float), stream);
            if (m == cudaSuccess) m = cudaMemsetAsync(a->dW3 + e * d * F, 0, (size_t)(d * F) * sizeof(float), stream);
            if (m == cudaSuccess) m = cudaMemsetAsync(a->dW2 + e * F * d, 0, (size_t)(F * d) * sizeof(float), stream);
            if (m != cudaSuccess) {
                (void)cudaGetLastError();
                return s3r_cuda_fail("ffn_backward: zeroing an empty expert's gradients", m);
            }
            continue;
        }
        const s3r_ffn_args g = expert_view(*a, e, r0, Tg);
        cur = (cur + 255) & ~(uintptr_t)255;
        const size_t need = layout(nullptr, 0, Tg, d, F, Tg, a->round_mode, fmt).total;
        if (cur + need > end) return S3R_ERR_WORKSPACE;
        blocks.emplace_back();
        S3R_TRY(make_block(blocks.back(), g, (void*)cur, need, (uint32_t)(S3R_MOE_TID_STRIDE * e)));
        cur += need;
    }
    const bool f16 = fmt == S3R_CODES_F16;
    const size_t nb = blocks.size();
    // The experts' EC passes on the side streams: blocks i and i + kSideStreams share a stream, so the
    // blocks of round i / kSideStreams run side by side; each takes a share of the SMs in proportion
    // to the codes it streams (weight side + its rows' input side), instead of all of them.
    {
        const int sms = s3r_sm_count();
        for (size_t r0 = 0; r0 < nb; r0 += kSideStreams) {
            const size_t r1 = std::min(nb, r0 + (size_t)kSideStreams);
            double w2 = 0.0, w13 = 0.0;
            for (size_t i = r0; i < r1; ++i) {
                w2 += (double)F * d + (double)blocks[i].a.T * F;
                w13 += 2.0 * d * F + (double)blocks[i].a.T * d;
            }
            for (size_t i = r0; i < r1; ++i) {
                const double my2 = (double)F * d + (double)blocks[i].a.T * F;
                const double my13 = 2.0 * d * F + (double)blocks[i].a.T * d;
                blocks[i].ec2_ctas = std::max(8, (int)(sms * my2 / w2));
                blocks[i].ec13_ctas = std::max(8, (int)(sms * my13 / w13));
            }
        }
    }
    S3R_TRY(record(a, 0, stream));
    S3R_TRY(run_on_side_streams(blocks, step_quantize_dy, stream));
    S3R_TRY(record(a, 1, stream));
    S3R_TRY(run_on_side_streams(blocks, step_ec_w2, stream));
    S3R_TRY(record(a, 2, stream));
    if (f16) {
        // dA and dW2 of every expert: mixed launches of up to MaxGroup / 2 experts
        const size_t per = MaxGroup / 2;
        for (size_t i0 = 0; i0 < nb; i0 += per) {
            UmmaDxProblem qx[MaxGroup / 2];
            UmmaDwProblem qw[MaxGroup / 2];
            const size_t n = std::min(nb - i0, per);
            for (size_t i = 0; i < n; ++i) {
                const Block& b = blocks[i0 + i];
                qx[i] = dx_problem_da(b);
                qw[i] = dw_problem(b, b.a.A8, b.Lo.w2, b.a.F, b.a.d, b.a.s_w2, b.a.dW2);
            }
            S3R_TRY(umma_mixed_group(qx, (int)n, qw, (int)n, a->d_status, stream));
        }
        S3R_TRY(record(a, 3, stream));
    } else {
        for (Block& b : blocks) S3R_TRY(step_da(b, stream));
        S3R_TRY(record(a, 3, stream));
        for (Block& b : blocks) S3R_TRY(step_dw2(b, stream));
    }
    S3R_TRY(record(a, 4, stream));
    S3R_TRY(run_on_side_streams(blocks, step_swiglu, stream));
    S3R_TRY(record(a, 5, stream));
    S3R_TRY(run_on_side_streams(blocks, step_ec_w13, stream));
    S3R_TRY(record(a, 6, stream));
    if (f16) {
        // dX1 + dX3, dW1 and dW3 of every expert: mixed launches of up to MaxGroup / 3 experts
        const size_t per = MaxGroup / 3;
        for (size_t i0 = 0; i0 < nb; i0 += per) {
            UmmaDxProblem qx[MaxGroup / 3];
            UmmaDwProblem qw[2 * (MaxGroup / 3)];
            const size_t n = std::min(nb - i0, per);
            for (size_t i = 0; i < n; ++i) {
                const Block& b = blocks[i0 + i];
                qx[i] = dx_problem_dx(b);
                qw[2 * i] = dw_problem(b, b.a.X8, b.Lo.w1, b.a.d, b.a.F, b.a.s_w1, b.a.dW1);
                qw[2 * i + 1] = dw_problem(b, b.a.X8, b.Lo.w3, b.a.d, b.a.F, b.a.s_w3, b.a.dW3);
            }
            S3R_TRY(umma_mixed_group(qx, (int)n, qw, (int)(2 * n), a->d_status, stream));
        }
        S3R_TRY(record(a, 7, stream));
    } else {
        for (Block& b : blocks) S3R_TRY(step_dx(b, stream));
        S3R_TRY(record(a, 7, stream));
        for (Block& b : blocks) S3R_TRY(step_dw13(b, stream));
    }
    return record(a, 8, stream);
}

// The block forward: RTNE operands (per-token X and a, per-output-channel
// weights), the gate and up projections in one launch (h1, h3 in bf16), the
// SwiGLU gate fused into the RTNE of a, then Y = a W2 in fp32 ("Efficient
// Quantization Training with Stochastic Rounding via Structured Subspace
// Randomness" §III-A, §IV-A).
extern "C" int ffn_forward(const struct s3r_ffn_fwd_args* a, cudaStream_t stream) {
    if (!a) return S3R_ERR_ARG;
    const int64_t T = a->T, d = a->d, F = a->F;
    if (T < 0 || d < 0 || F < 0) return S3R_ERR_ARG;
    if (a->code_format != S3R_CODES_F16) {
        s3r_record_error("ffn_forward", "the forward runs on fp16-carried codes (S3R_CODES_F16) only");
        return S3R_ERR_UNSUPPORTED;
    }
    if (T == 0 || d == 0 || F == 0) return S3R_OK;
    if (!a->X || !a->X8 || !a->s_x || !a->W1_8 || !a->s_w1 || !a->W3_8 || !a->s_w3 || !a->W2_8 || !a->s_w2 ||
        !a->h1 || !a->h3 || !a->A8 || !a->s_a || !a->Y)
        return S3R_ERR_ARG;
    if (a->quantize_weights && (!a->W1 || !a->W3 || !a->W2)) return S3R_ERR_ARG;
    const int fmt = S3R_CODES_F16;
    S3R_TRY(rtne_quantize(a->X, T, d, d, nullptr, nullptr, S3R_AXIS_ROW, a->X8, fmt, a->s_x, a->d_status, stream));
    if (a->quantize_weights) {
        S3R_TRY(rtne_quantize(a->W1, d, F, F, nullptr, nullptr, S3R_AXIS_COL, a->W1_8, fmt, a->s_w1, a->d_status,
                              stream));
        S3R_TRY(rtne_quantize(a->W3, d, F, F, nullptr, nullptr, S3R_AXIS_COL, a->W3_8, fmt, a->s_w3, a->d_status,
                              stream));
        S3R_TRY(rtne_quantize(a->W2, F, d, d, nullptr, nullptr, S3R_AXIS_COL, a->W2_8, fmt, a->s_w2, a->d_status,
                              stream));
    }
    S3R_TRY(int8_gemm_fwd_swiglu(a->X8, a->s_x, a->W1_8, a->s_w1, a->W3_8, a->s_w3, fmt, T, d, F, a->h1, a->h3,
                                 nullptr, a->d_status, stream));
    S3R_TRY(swiglu_fwd_quantize(a->h1, a->h3, T, F, F, a->a, a->A8, fmt, a->s_a, a->d_status, stream));
    return int8_gemm_fwd(a->A8, a->s_a, a->W2_8, a->s_w2, fmt, T, F, d, a->Y, a->d_status, stream);
}

extern "C" const char* s3r_status_string(int status) {
    switch (status) {
        case S3R_OK: return "S3R_OK";
        case S3R_ERR_ARG: return "S3R_ERR_ARG: invalid argument";
        case S3R_ERR_ALIGN: return "S3R_ERR_ALIGN: pointer or stride not 16-byte aligned";
        case S3R_ERR_SHAPE: return "S3R_ERR_SHAPE: inconsistent sizes";
        case S3R_ERR_NONFINITE: return "S3R_ERR_NONFINITE: NaN or Inf in the folded gradient";
        case S3R_ERR_TIMEOUT: return "S3R_ERR_TIMEOUT: a bounded device wait gave up";
        case S3R_ERR_CUDA: return "S3R_ERR_CUDA: CUDA launch or attribute call failed";
        case S3R_ERR_WORKSPACE: return "S3R_ERR_WORKSPACE: workspace missing or too small";
        case S3R_ERR_UNSUPPORTED: return "S3R_ERR_UNSUPPORTED: size outside the supported range";
        default: return "S3R_ERR_UNKNOWN";
    }
}

extern "C" int s3r_abi_version(void) { return 104; }
