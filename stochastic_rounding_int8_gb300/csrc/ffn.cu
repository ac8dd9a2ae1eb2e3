// ffn.cu -- SwiGLU FFN block backward built from the library's entry points,
// and the status helpers.
//
// Paper: "Efficient Quantization Training with Stochastic Rounding via
// Structured Subspace Randomness" §IV-A (single-block SwiGLU FFN benchmark,
// Table III shapes), §III-A..§III-D for each linear.  One stream, no host
// synchronization; every intermediate lives in the caller's workspace.
#include <atomic>

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

namespace {

constexpr uint32_t kRhsOffset = S3R_TID_RHS_OFFSET;

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

extern "C" size_t s3r_ffn_workspace_size(int64_t T, int64_t d, int64_t F, int64_t S, int round_mode, int ec_mode,
                                         int code_format) {
    (void)ec_mode;
    if (T <= 0 || d <= 0 || F <= 0 || S <= 0 || T % S != 0) return 0;
    return layout(nullptr, 0, T, d, F, S, round_mode, code_format).total;
}

namespace {

// The block backward of one example group (the whole batch, or one expert's
// rows): a->T rows, a->S tokens per example, tensor ids tid_base + (0, 1, 2).
// Step events are recorded only when `events` is set.
int run_block(const struct s3r_ffn_args* a, uint32_t tid_base, bool events, cudaStream_t stream) {
    const int64_t T = a->T, d = a->d, F = a->F, S = a->S;
    const int fmt = a->code_format;
    FfnLayout Lo = layout(a->workspace, a->workspace_bytes, T, d, F, S, a->round_mode, fmt);
    if (!Lo.ok) return S3R_ERR_WORKSPACE;
    const int rm = a->round_mode;
    const int ec = rm == S3R_ROUND_S3R ? a->ec_mode : S3R_EC_NONE;
    const bool indep = rm == S3R_ROUND_INDEP;
    const uint32_t kTidW2 = tid_base + S3R_TID_W2, kTidW1 = tid_base + S3R_TID_W1, kTidW3 = tid_base + S3R_TID_W3;
    int* st = a->d_status;
    auto mark = [&](int i) -> int {
        if (events && a->step_events) {
            cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(a->step_events[i]), stream);
            if (e != cudaSuccess) {
                (void)cudaGetLastError();
                return s3r_cuda_fail("ffn_backward step event", e);
            }
        }
        return S3R_OK;
    };
    S3R_TRY(mark(0));

    // 1. quantize dY with the W2 fold (s_a per token, s_w2 per output channel)
    LinearWs& L2 = Lo.w2;
    if (rm == S3R_ROUND_S3R) {
        S3R_TRY(s3r_quantize(a->dY, T, d, d, a->s_a, a->s_w2, a->seed, kTidW2, L2.Q, fmt, L2.scale, L2.tok, L2.col,
                             st, stream));
    } else if (indep) {
        S3R_TRY(indep_sr_quantize(a->dY, T, d, d, a->s_a, a->s_w2, a->seed, kTidW2, L2.Q, fmt, L2.scale, st, stream));
        S3R_TRY(indep_sr_quantize(a->dY, T, d, d, a->s_a, a->s_w2, a->seed, kTidW2 + kRhsOffset, L2.Qr, fmt,
                                  L2.scale_r, st, stream));
    } else {
        S3R_TRY(rtne_quantize(a->dY, T, d, d, a->s_a, a->s_w2, S3R_AXIS_TILE, L2.Q, fmt, L2.scale, st, stream));
    }
    S3R_TRY(mark(1));
    // 2. correction factors of W2 (W8 = W2_8 [F, d], X8 = A8 [T, F])
    if (ec != S3R_EC_NONE)
        S3R_TRY(s3r_ec_correct(L2.tok, L2.col, T, d, S, a->W2_8, F, a->A8, fmt, ec, L2.eps, L2.mu, L2.colmean,
                               L2.rowsum, L2.v, L2.xsum, L2.p, Lo.ec_ws, Lo.ec_ws_bytes, st, stream));
    S3R_TRY(mark(2));
    // 3. dA = Q2 W2_8^T (rescaled, corrected, / s_a)  [T, F]
    S3R_TRY(int8_gemm_dx(L2.Q, L2.scale, a->W2_8, fmt, T, d, F, a->s_a, ec, L2.eps, L2.rowsum, L2.v, S, Lo.dA, 0,
                         st, stream));
    S3R_TRY(mark(3));
    // 4. dW2 = A8^T Q2 / s_w2  [F, d]
    S3R_TRY(int8_gemm_dw(a->A8, indep ? L2.Qr : L2.Q, indep ? L2.scale_r : L2.scale, fmt, T, F, d, a->s_w2, ec,
                         L2.colmean, L2.mu, L2.xsum, L2.p, S, a->dW2, Lo.dw_ws, Lo.dw_ws_bytes, st, stream));
    S3R_TRY(mark(4));
    // 5. SwiGLU glue fused into the quantization of dh1 (W1 fold) and dh3 (W3 fold)
    LinearWs &L1 = Lo.w1, &L3 = Lo.w3;
    const bool keep_err = ec != S3R_EC_NONE;
    S3R_TRY(swiglu_quantize(Lo.dA, F, a->h1, a->h3, F, T, F, a->s_x, a->s_w1, a->s_w3, rm, fmt, a->seed, kTidW1,
                            kTidW3, L1.Q, L1.scale, keep_err ? L1.tok : nullptr, keep_err ? L1.col : nullptr, L3.Q,
                            L3.scale, keep_err ? L3.tok : nullptr, keep_err ? L3.col : nullptr, st, stream));
    if (indep)
        S3R_TRY(swiglu_quantize(Lo.dA, F, a->h1, a->h3, F, T, F, a->s_x, a->s_w1, a->s_w3, rm, fmt, a->seed,
                                kTidW1 + kRhsOffset, kTidW3 + kRhsOffset, L1.Qr, L1.scale_r, nullptr, nullptr, L3.Qr,
                                L3.scale_r, nullptr, nullptr, st, stream));
    S3R_TRY(mark(5));
    // 6. correction factors of W1 and W3 (W8 [d, F], X8 [T, d])
    if (ec != S3R_EC_NONE) {
        S3R_TRY(s3r_ec_correct_pair(L1.tok, L1.col, a->W1_8, L1.eps, L1.mu, L1.colmean, L1.rowsum, L1.v, L1.xsum,
                                    L1.p, L3.tok, L3.col, a->W3_8, L3.eps, L3.mu, L3.colmean, L3.rowsum, L3.v,
                                    L3.xsum, L3.p, T, F, S, d, a->X8, fmt, ec, Lo.ec_ws, Lo.ec_ws_bytes, stream));
    }
    S3R_TRY(mark(6));
    // 7. dX = dX1 + dX3
    const s3r_dx_term terms[2] = {{L1.Q, L1.scale, a->W1_8, L1.eps, L1.rowsum, L1.v},
                                  {L3.Q, L3.scale, a->W3_8, L3.eps, L3.rowsum, L3.v}};
    S3R_TRY(int8_gemm_dx_sum(terms, 2, fmt, T, F, d, a->s_x, ec, S, a->dX, 0, st, stream));
    S3R_TRY(mark(7));
    // 8. dW1, dW3
    if (fmt == S3R_CODES_F16) {
        // both weight gradients in one persistent launch (their tiles share the grid)
        const bool two = ec == S3R_EC_TWO_WAY;
        const UmmaDwProblem q[2] = {
            {a->X8, indep ? L1.Qr : L1.Q, indep ? L1.scale_r : L1.scale, T, d, F, a->s_w1, ec,
             two ? L1.colmean : nullptr, two ? L1.mu : nullptr, two ? L1.xsum : nullptr, two ? L1.p : nullptr, S,
             a->dW1, nullptr},
            {a->X8, indep ? L3.Qr : L3.Q, indep ? L3.scale_r : L3.scale, T, d, F, a->s_w3, ec,
             two ? L3.colmean : nullptr, two ? L3.mu : nullptr, two ? L3.xsum : nullptr, two ? L3.p : nullptr, S,
             a->dW3, nullptr}};
        S3R_TRY(umma_dw_group(q, 2, st, stream));
    } else {
        S3R_TRY(int8_gemm_dw(a->X8, indep ? L1.Qr : L1.Q, indep ? L1.scale_r : L1.scale, fmt, T, d, F, a->s_w1, ec,
                             L1.colmean, L1.mu, L1.xsum, L1.p, S, a->dW1, Lo.dw_ws, Lo.dw_ws_bytes, st, stream));
        S3R_TRY(int8_gemm_dw(a->X8, indep ? L3.Qr : L3.Q, indep ? L3.scale_r : L3.scale, fmt, T, d, F, a->s_w3, ec,
                             L3.colmean, L3.mu, L3.xsum, L3.p, S, a->dW3, Lo.dw_ws, Lo.dw_ws_bytes, st, stream));
    }
    S3R_TRY(mark(8));
    return S3R_OK;
}

}  // namespace

extern "C" int ffn_backward(const struct s3r_ffn_args* a, cudaStream_t stream) {
    if (!a) return S3R_ERR_ARG;
    const int64_t T = a->T, d = a->d, F = a->F, S = a->S;
    if (T <= 0 || d <= 0 || F <= 0) return S3R_ERR_ARG;
    if (a->round_mode < S3R_ROUND_RTNE || a->round_mode > S3R_ROUND_INDEP) return S3R_ERR_ARG;
    if (a->ec_mode < S3R_EC_NONE || a->ec_mode > S3R_EC_TWO_WAY) return S3R_ERR_ARG;
    if (a->code_format != S3R_CODES_S8 && a->code_format != S3R_CODES_F16) return S3R_ERR_ARG;
    const int fmt = a->code_format;
    if (!a->dY || !a->h1 || !a->h3 || !a->X8 || !a->A8 || !a->W1_8 || !a->W3_8 || !a->W2_8 || !a->dX || !a->dW1 ||
        !a->dW2 || !a->dW3)
        return S3R_ERR_ARG;
    if (a->num_groups == 0) {
        if (S <= 0) return S3R_ERR_ARG;
        if (T % S != 0 || (S % S3R_TILE != 0 && S != T)) return S3R_ERR_SHAPE;
        if (!a->workspace || a->workspace_bytes < s3r_ffn_workspace_size(T, d, F, S, a->round_mode, a->ec_mode, fmt))
            return S3R_ERR_WORKSPACE;
        return run_block(a, 0, true, stream);
    }
    // grouped: expert e owns rows offsets[e] .. offsets[e+1] (one example);
    // weights, their scales and gradients are stacked per expert
    const int64_t E = a->num_groups;
    const int64_t* off = a->group_offsets;
    if (E < 0 || !off || off[0] != 0 || off[E] != T) return S3R_ERR_ARG;
    int64_t tmax = 0;
    for (int64_t e = 0; e < E; ++e) {
        if (off[e + 1] < off[e]) return S3R_ERR_ARG;
        tmax = off[e + 1] - off[e] > tmax ? off[e + 1] - off[e] : tmax;
    }
    if (E > (int64_t)(0xFFFFFFFFu / S3R_MOE_TID_STRIDE)) return S3R_ERR_ARG;
    if (!a->workspace ||
        a->workspace_bytes < s3r_ffn_workspace_size(tmax, d, F, tmax, a->round_mode, a->ec_mode, fmt))
        return S3R_ERR_WORKSPACE;
    const size_t cs = fmt == S3R_CODES_F16 ? 2 : 1;
    if (a->step_events) {
        cudaError_t ev = cudaEventRecord(static_cast<cudaEvent_t>(a->step_events[0]), stream);
        if (ev != cudaSuccess) {
            (void)cudaGetLastError();
            return s3r_cuda_fail("ffn_backward step event", ev);
        }
    }
    for (int64_t e = 0; e < E; ++e) {
        const int64_t r0 = off[e], Tg = off[e + 1] - off[e];
        float* dW1 = a->dW1 + e * d * F;
        float* dW3 = a->dW3 + e * d * F;
        float* dW2 = a->dW2 + e * F * d;
        if (Tg == 0) {   // an expert without rows has zero weight gradients
            cudaError_t m = cudaMemsetAsync(dW1, 0, (size_t)(d * F) * sizeof(float), stream);
            if (m == cudaSuccess) m = cudaMemsetAsync(dW3, 0, (size_t)(d * F) * sizeof(float), stream);
            if (m == cudaSuccess) m = cudaMemsetAsync(dW2, 0, (size_t)(F * d) * sizeof(float), stream);
            if (m != cudaSuccess) {
                (void)cudaGetLastError();
                return s3r_cuda_fail("ffn_backward: zeroing an empty expert's gradients", m);
            }
            continue;
        }
        s3r_ffn_args g = *a;
        g.T = Tg;
        g.S = Tg;
        g.num_groups = 0;
        g.group_offsets = nullptr;
        g.dY = static_cast<const uint16_t*>(a->dY) + r0 * d;
        g.h1 = static_cast<const uint16_t*>(a->h1) + r0 * F;
        g.h3 = static_cast<const uint16_t*>(a->h3) + r0 * F;
        g.X8 = static_cast<const uint8_t*>(a->X8) + (size_t)(r0 * d) * cs;
        g.s_x = a->s_x ? a->s_x + r0 : nullptr;
        g.A8 = static_cast<const uint8_t*>(a->A8) + (size_t)(r0 * F) * cs;
        g.s_a = a->s_a ? a->s_a + r0 : nullptr;
        g.W1_8 = static_cast<const uint8_t*>(a->W1_8) + (size_t)(e * d * F) * cs;
        g.s_w1 = a->s_w1 ? a->s_w1 + e * F : nullptr;
        g.W3_8 = static_cast<const uint8_t*>(a->W3_8) + (size_t)(e * d * F) * cs;
        g.s_w3 = a->s_w3 ? a->s_w3 + e * F : nullptr;
        g.W2_8 = static_cast<const uint8_t*>(a->W2_8) + (size_t)(e * F * d) * cs;
        g.s_w2 = a->s_w2 ? a->s_w2 + e * d : nullptr;
        g.dX = a->dX + r0 * d;
        g.dW1 = dW1;
        g.dW3 = dW3;
        g.dW2 = dW2;
        S3R_TRY(run_block(&g, (uint32_t)(S3R_MOE_TID_STRIDE * e), false, stream));
    }
    if (a->step_events) {
        for (int i = 1; i < S3R_FFN_NUM_EVENTS; ++i) {
            cudaError_t ev = cudaEventRecord(static_cast<cudaEvent_t>(a->step_events[i]), stream);
            if (ev != cudaSuccess) {
                (void)cudaGetLastError();
                return s3r_cuda_fail("ffn_backward step event", ev);
            }
        }
    }
    return S3R_OK;
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

extern "C" int s3r_abi_version(void) { return 100; }
