/*
 * s3r.h -- C ABI of libs3r, a GB300 (sm_103a) implementation of the S3R /
 * S3R-EC INT8 backward pass of a linear or SwiGLU FFN layer, the INT8
 * forward of the same block, and stochastic rounding of fp32 to bf16 / FP8
 * with the same shared thresholds.
 *
 * Entry points: quantizers (s3r_quantize, s3r_quantize_ex, indep_sr_quantize,
 * rtne_quantize, swiglu_quantize, swiglu_quantize_ex, swiglu_fwd_quantize),
 * correction factors (s3r_ec_correct, s3r_ec_correct_static), products
 * (int8_gemm_dx, int8_gemm_dx_sum, int8_gemm_dw, int8_gemm_fwd,
 * int8_gemm_fwd_swiglu), whole block (ffn_backward, ffn_forward), SR to
 * floating point (s3r_sr_bf16, s3r_sr_fp8), status and debug helpers.
 *
 * Method: "Efficient Quantization Training with Stochastic Rounding via
 * Structured Subspace Randomness" (cited below as [S3R] with its sections:
 * §III-A quantized backprop with SR, §III-B structured subspace randomness,
 * §III-C why sharing hurts, §III-D S3R-EC, §IV-B compared configurations).
 * SR definition: "Stochastic Rounding" (transformer-math blog), sections
 * "Stochastic rounding, defined" and "The probability formula".
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Notation: a linear layer Y = X W with X [T, K] (T = B*S tokens, B
 *    examples of S tokens), W [K, N], upstream gradient G = dY [T, N].
 *  - All tensors are row-major.  "ld*" arguments are row strides in elements.
 *    bf16 tensors are passed as `const void*` holding IEEE bfloat16.
 *  - Every pointer except those documented as host pointers is a DEVICE
 *    pointer owned by the caller.  The library never allocates device memory
 *    and never synchronizes; where scratch is needed the caller passes a
 *    workspace whose size a *_workspace_size() call returns.
 *  - Every call is asynchronous on `stream` and returns an int status
 *    (S3R_OK = 0, negative on error) for what the host can check: null or
 *    misaligned pointers, bad sizes, launch failures.  Nothing is launched
 *    when the host check fails.  Conditions only the device can see (a
 *    non-finite gradient value, a bounded wait that ran out) are written to
 *    `d_status` (a device int, may be NULL), which the caller reads after
 *    synchronizing; the call itself then still returns S3R_OK.  The caller
 *    zeroes *d_status before the first call; calls only ever write error
 *    codes into it.
 *  - Tiles are S3R_TILE x S3R_TILE = 128 x 128 and start at row 0 and column 0;
 *    the last tile row / column may be partial (ragged T and N are allowed).
 *  - Base pointers of int8 and bf16 tensors must be 16-byte aligned and their
 *    row strides multiples of 16 bytes (S3R_ERR_ALIGN otherwise).
 *  - No exception crosses the ABI.
 */
#ifndef S3R_H
#define S3R_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same definition as the CUDA runtime's. */
typedef struct CUstream_st* cudaStream_t;

#define S3R_TILE 128

enum s3r_status {
    S3R_OK = 0,
    S3R_ERR_ARG = -1,        /* null pointer, negative size, unknown enum */
    S3R_ERR_ALIGN = -2,      /* base pointer or row stride not 16-byte aligned */
    S3R_ERR_SHAPE = -3,      /* inconsistent sizes (e.g. T not a multiple of S) */
    S3R_ERR_NONFINITE = -4,  /* (device) NaN or Inf in the folded gradient */
    S3R_ERR_TIMEOUT = -5,    /* (device) a bounded wait gave up */
    S3R_ERR_CUDA = -6,       /* a CUDA launch or attribute call failed */
    S3R_ERR_WORKSPACE = -7,  /* workspace null or smaller than required */
    S3R_ERR_UNSUPPORTED = -8 /* size outside what the kernels support */
};

/* Error correction ([S3R] §III-D). */
enum s3r_ec_mode {
    S3R_EC_NONE = 0,     /* plain S3R (or a baseline rounding) */
    S3R_EC_DX_ONLY = 1,  /* subtract P(E) W^T from the activation gradient only */
    S3R_EC_TWO_WAY = 2,  /* also subtract X^T P(E) from the weight gradient */
    S3R_EC_DW_ONLY = 3   /* ablation ([S3R] Table II): the weight-gradient term only */
};

/* How the upstream gradient is rounded ([S3R] §IV-B). */
enum s3r_round_mode {
    S3R_ROUND_RTNE = 0,  /* deterministic round to nearest even */
    S3R_ROUND_S3R = 1,   /* one threshold per token shared by its channels (Phi_2D) */
    S3R_ROUND_INDEP = 2, /* one threshold per element (conventional SR) */
    /* [S3R] §III-B, the paper's own thresholds: Phi_2D with 7-bit values, four cut
     * from each 32-bit word (token t: upper 7 bits k of byte t mod 4 of word 0 of
     * Philox(counter = t / 4)), on the grid shifted by half a step, u = (k + 1/2)/128;
     * the rounding bias is at most Delta/256. */
    S3R_ROUND_S3R_7BIT = 3,
    /* [S3R] §III-B, Phi_bcast (ablation): one threshold per example of S tokens,
     * word 0 of Philox(counter = (b, 0, 1, 0)) on the 24-bit grid */
    S3R_ROUND_BCAST = 4
};

/* Storage of the integer codes (values in [-127, 127]).  S8 is one byte per
 * code.  F16 stores the same integer exactly in an IEEE half: sm_103a has no
 * integer tcgen05 MMA and its warp-level s8 MMA runs far below the 16-bit
 * tensor rate, so F16 is the operand format of the tensor-core GEMMs here
 * (TMA straight into the MMA's shared-memory layout, no conversion pass).
 * Both products of one layer must use the same format. */
enum s3r_code_format {
    S3R_CODES_S8 = 0,     /* int8_t [rows, cols] */
    S3R_CODES_F16 = 1,    /* IEEE fp16 [rows, cols], integer valued; cols % 8 == 0 for the GEMMs */
    S3R_CODES_S8_F16 = 2  /* ffn_backward only: the operand codes at rest as int8_t (half the bytes
                             of F16), widened to fp16 inside the call; computed as F16 */
};

/* Scale granularity of rtne_quantize. */
enum s3r_scale_axis {
    S3R_AXIS_ROW = 0,  /* one scale per row:    A ~= diag(s) A_hat (per-token s_x) */
    S3R_AXIS_COL = 1,  /* one scale per column: A ~= A_hat diag(s) (per-channel s_w) */
    S3R_AXIS_TILE = 2  /* one scale per 128x128 tile (RTNE baseline for dY) */
};

/* Human-readable name of a status code (static string, never NULL). */
const char* s3r_status_string(int status);

/* ABI version of this header (major*100 + minor). */
int s3r_abi_version(void);

/* Number of kernels this library has launched in this process (a host-side
 * count, for measurement). */
uint64_t s3r_kernel_launch_count(void);

/* Description of the last failure this thread saw (which call, and the CUDA
 * error or the tensor-map encoder's result); "" when none.  Static per-thread
 * storage, valid until the thread's next failing call. */
const char* s3r_last_error(void);

/*
 * s3r_quantize -- S3R quantization of the upstream gradient, written once for
 * both backward products ([S3R] §III-A eq. (2) "fold and quantize once",
 * §III-B inter-operand sharing and per-token threshold broadcast Phi_2D).
 *
 * For every element, in fp32 and in this order:
 *   g    = (s_x[t] * G[t,n]) * s_w[n]     fold; a NULL scale pointer means 1
 *   amax = max |g| over its 128x128 tile;  tile_scale = amax / 127
 *   y    = g * (127 / amax)               (y = 0 when amax = 0)
 *   u_t  = (w >> 8) * 2^-24, w = word 0 of Philox4x32-10 with
 *          counter (t mod 2^32, t >> 32, 0, 0), key (seed mod 2^32, tensor_id)
 *   q    = clamp(floor(y) + [u_t < y - floor(y)], -127, 127)
 *   e    = fma(tile_scale, q, -g)         the rounding error E = Delta Q - G'
 *
 * In : G [T, N] bf16 (row stride ldg >= N); s_x [T] or NULL; s_w [N] or NULL.
 * Out: Q [T, N] codes in `code_format` (row stride N); tile_scale [ceil(T/128), ceil(N/128)];
 *      tok_err_part [T, ceil(N/128)]  sum of e over each tile's columns, per token;
 *      col_err_part [ceil(T/128), N]  sum of e over each tile's rows, per channel.
 *      Both partial arrays may be NULL (then they are not written).
 * A tile holding a non-finite g gets tile_scale = NaN, Q = 0, zero partials and
 * sets *d_status = S3R_ERR_NONFINITE.
 */
int s3r_quantize(const void* G, int64_t T, int64_t N, int64_t ldg, const float* s_x, const float* s_w,
                 uint64_t seed, uint32_t tensor_id, void* Q, int code_format, float* tile_scale,
                 float* tok_err_part, float* col_err_part, int* d_status, cudaStream_t stream);

/*
 * s3r_quantize_ex -- s3r_quantize with the paper's own variants ([S3R] §III-A,
 * §III-B): any `round_mode` (s3r_round_mode), S tokens per example (the
 * examples of S3R_ROUND_BCAST; 0 = one example; T % S == 0 otherwise), and an
 * optional per-tensor step.  With tensor_amax non-NULL (a device float) the
 * call first sets *tensor_amax = max |g| over the whole tensor and then uses
 * amax / 127 as the step of every tile: every tile_scale entry holds that
 * step, which is [S3R]'s Delta = max|G'|/127.  The error partials are written
 * for the shared-threshold modes (S3R, S3R_7BIT, BCAST) and left untouched
 * otherwise.  Everything else is as in s3r_quantize.
 */
int s3r_quantize_ex(const void* G, int64_t T, int64_t N, int64_t ldg, const float* s_x, const float* s_w,
                    int round_mode, int64_t S, float* tensor_amax, uint64_t seed, uint32_t tensor_id, void* Q,
                    int code_format, float* tile_scale, float* tok_err_part, float* col_err_part, int* d_status,
                    cudaStream_t stream);

/*
 * indep_sr_quantize -- conventional stochastic rounding with an independent
 * threshold per element ([S3R] §III-A, "Conventional QT implementations draw
 * independent full-size thresholds"; §IV-B "Independent SR").  Same fold, tile
 * scale, clamp and layout as s3r_quantize; the threshold of element
 * e = t*N + n is word (e mod 4) of Philox4x32-10 with counter
 * (floor(e/4) mod 2^32, floor(e/4) >> 32, 0, 0) and key (seed mod 2^32,
 * tensor_id).  Call it twice with two tensor ids for the two products.
 */
int indep_sr_quantize(const void* G, int64_t T, int64_t N, int64_t ldg, const float* s_x, const float* s_w,
                      uint64_t seed, uint32_t tensor_id, void* Q, int code_format, float* tile_scale,
                      int* d_status, cudaStream_t stream);

/*
 * rtne_quantize -- round to nearest even ([S3R] §III-A forward operands;
 * §IV-B "INT8 RTNE").  q = clamp(rint(a * (127 / amax)), -127, 127) with
 * amax taken per row, per column or per 128x128 tile of the folded input
 * a = (s_x[r] * A[r,c]) * s_w[c] (NULL scale = 1).
 * Out: Q [R, C] codes in `code_format` (row stride C); scale = amax / 127 per row [R], per
 * column [C] or per tile [ceil(R/128), ceil(C/128)].  For ROW and COL an
 * all-zero row/column gets scale 1 (any scale reproduces zero; 1 keeps the
 * backward fold finite); for TILE an all-zero tile gets scale 0.
 */
int rtne_quantize(const void* A, int64_t R, int64_t C, int64_t lda, const float* s_x, const float* s_w,
                  int scale_axis, void* Q, int code_format, float* scale, int* d_status, cudaStream_t stream);

/*
 * swiglu_quantize -- the SwiGLU backward glue fused into the quantization of
 * the two gate/up gradients (FFN block of [S3R] §IV-A).  With a = silu(h1)*h3
 * and dA = dL/da, in fp32 and in this order:
 *   s = sigmoid(h1) = 1 / (1 + exp(-h1)),  silu = h1*s,
 *   dsilu = s * (1 + h1*(1 - s)),  dh1 = (dA*h3) * dsilu,  dh3 = dA * silu,
 * where exp is Cody-Waite reduction (ln 2 split in a 16-bit head and a tail)
 * with a degree-7 Taylor polynomial and the argument clamped to [-87, 88].
 * dh1 and dh3 are then quantized exactly as s3r_quantize would quantize them
 * (fold with s_x [T] and s_w1 / s_w3 [F]), with `round_mode` choosing the
 * rounding (s3r_round_mode) and tensor ids tid1 / tid3.
 * In : dA [T, F] fp32 (row stride ldd); h1, h3 [T, F] bf16 (row stride ldh).
 * Out: Q1, Q3 [T, F] codes in `code_format`; scale1, scale3 tile scales; tok1/col1/tok3/col3
 *      error partials as in s3r_quantize (NULL allowed).
 */
int swiglu_quantize(const float* dA, int64_t ldd, const void* h1, const void* h3, int64_t ldh, int64_t T,
                    int64_t F, const float* s_x, const float* s_w1, const float* s_w3, int round_mode,
                    int code_format, uint64_t seed, uint32_t tid1, uint32_t tid3, void* Q1, float* scale1,
                    float* tok1, float* col1, void* Q3, float* scale3, float* tok3, float* col3, int* d_status,
                    cudaStream_t stream);
/* swiglu_quantize_ex -- the same with S tokens per example for S3R_ROUND_BCAST
 * (0 = one example; T % S == 0 otherwise). */
int swiglu_quantize_ex(const float* dA, int64_t ldd, const void* h1, const void* h3, int64_t ldh, int64_t T,
                       int64_t F, const float* s_x, const float* s_w1, const float* s_w3, int round_mode, int64_t S,
                       int code_format, uint64_t seed, uint32_t tid1, uint32_t tid3, void* Q1, float* scale1,
                       float* tok1, float* col1, void* Q3, float* scale3, float* tok3, float* col3, int* d_status,
                       cudaStream_t stream);

/*
 * s3r_ec_correct -- the error statistics and correction factors of S3R-EC
 * ([S3R] §III-D, "Two-way correction").  With e the rounding error of
 * s3r_quantize and example b the S consecutive tokens [b*S, (b+1)*S):
 *   eps[t]        = (1/N) sum_n e[t,n]                 token mean
 *   colmean[b,n]  = (1/S) sum_{t in b} e[t,n]          channel mean of example b
 *   mu[b]         = (1/(S*N)) sum_{t in b, n} e[t,n]   grand mean
 * so that P(E_b) = 1 colmean_b^T + eps_b 1^T - mu_b 1 1^T is the orthogonal
 * projection onto row- and column-constant matrices, and
 *   rowsum[k]     = sum_n W8[k,n]                      (W 1_D)
 *   v[b,k]        = sum_n (colmean[b,n] - mu[b]) W8[k,n]
 * and for S3R_EC_TWO_WAY also
 *   xsum[b,k]     = sum_{t in b} X8[t,k]
 *   p[k]          = sum_t X8[t,k] eps[t].
 * In : the partial sums from s3r_quantize; W8 [K, N] and X8 [T, K] codes in
 *      `code_format` (X8 two-way only, else may be NULL).  Requires T % S == 0 and either
 *      S % 128 == 0 or S == T.
 * Out: eps [T], mu [B], colmean [B, N], rowsum [K] int32, v [B, K];
 *      two-way: xsum [B, K] int32, p [K].
 * workspace: s3r_ec_workspace_size(T, K) bytes (two-way and dW-only; else may be NULL).
 */
size_t s3r_ec_workspace_size(int64_t T, int64_t K);
int s3r_ec_correct(const float* tok_err_part, const float* col_err_part, int64_t T, int64_t N, int64_t S,
                   const void* W8, int64_t K, const void* X8, int code_format, int ec_mode, float* eps, float* mu,
                   float* colmean, int32_t* rowsum, float* v, int32_t* xsum, float* p, void* workspace,
                   size_t workspace_bytes, int* d_status, cudaStream_t stream);

/*
 * s3r_ec_correct_static -- s3r_ec_correct without a caller workspace, for
 * callers that cannot allocate device memory when they run it (from a host
 * callback or a real-time loop, where an allocation may block or fail, or
 * under a device memory budget fixed before the first step).  The
 * paper has no counterpart: this is a deployment convenience of this library.
 * Arguments and results are those of s3r_ec_correct.  The two-way column sums
 * use a scratch array of 8 MiB that lives in the library (every GPU that loads
 * the library keeps it until the process exits); sizes whose scratch
 * (s3r_ec_workspace_size(T, K)) exceeds 8 MiB are rejected with
 * S3R_ERR_UNSUPPORTED and an explanation in s3r_last_error().  The first call
 * on a device looks up the array's device address; make that first call before
 * any stream capture.  Every call shares the array, so calls that overlap on
 * the GPU (other streams or threads) race on it.  Allocates nothing.
 */
int s3r_ec_correct_static(const float* tok_err_part, const float* col_err_part, int64_t T, int64_t N, int64_t S,
                          const void* W8, int64_t K, const void* X8, int code_format, int ec_mode, float* eps,
                          float* mu, float* colmean, int32_t* rowsum, float* v, int32_t* xsum, float* p,
                          int* d_status, cudaStream_t stream);

/*
 * int8_gemm_dx -- activation gradient from the S8 codes ([S3R] §III-A "S8 GEMM
 * with S32 accumulation, and rescaled"; §III-D activation-gradient term):
 *   acc[t,k] = sum_kb tile_scale[t/128, kb] * (int32) sum_{n in block kb} Q[t,n] W8[k,n]
 *   dX[t,k]  = (acc - eps[t]*rowsum[k] - v[t/S, k]) / s_x[t]     (EC modes 1, 2)
 *   dX[t,k]  = acc / s_x[t]                                      (EC mode 0)
 * (plus the old dX[t,k] when accumulate != 0).  Each 128-wide block is an
 * exact integer; blocks are combined in fp32.  S3R_CODES_F16 runs on tcgen05
 * (kind::f16, fp32 accumulator drained per block; needs N % 8 == 0);
 * S3R_CODES_S8 runs on the warp-level s8 mma.sync path.
 * In : Q [T, N] codes; tile_scale from the quantizer; W8 [K, N] codes (the
 *      forward weight's codes, W [K, N] ~= W8 diag(s_w)); s_x [T] or NULL;
 *      eps, rowsum, v from s3r_ec_correct (unused when ec_mode = 0).
 * Out: dX [T, K] fp32 (row stride K).
 */
int int8_gemm_dx(const void* Q, const float* tile_scale, const void* W8, int code_format, int64_t T, int64_t N,
                 int64_t K, const float* s_x, int ec_mode, const float* eps, const int32_t* rowsum, const float* v,
                 int64_t S, float* dX, int accumulate, int* d_status, cudaStream_t stream);

/*
 * int8_gemm_dx_sum -- activation gradient of a layer whose input feeds several
 * linears, dX = sum_i (corrected, rescaled) Q_i W8_i^T.  The SwiGLU FFN block
 * of [S3R] §IV-A (Table III) feeds X to both W1 and W3, so its input gradient
 * is dX1 + dX3; each term follows the int8_gemm_dx formula with its own codes,
 * tile scales and correction, and all terms share T, N, K, s_x and ec_mode:
 *   dX[t,k] = (sum_i (acc_i - eps_i[t]*rowsum_i[k] - v_i[t/S, k])) / s_x[t]
 * (plus the old dX when accumulate != 0).  S3R_CODES_F16 contracts every term
 * into one fp32 accumulator in a single tcgen05 launch (one rescale, one store
 * of dX); S3R_CODES_S8 runs one int8_gemm_dx per term, the later ones
 * accumulating, so the two formats round the sum in a different order.
 * terms: HOST array of n_terms (1 .. S3R_DX_MAX_TERMS) entries, read during
 *        the call only; every pointer in it is a device pointer as in
 *        int8_gemm_dx (eps, rowsum, v may be NULL when ec_mode = 0).
 * Out: dX [T, K] fp32 (row stride K).
 */
#define S3R_DX_MAX_TERMS 2
struct s3r_dx_term {
    const void* Q;               /* [T, N] codes of this term's gradient */
    const float* tile_scale;     /* its per-tile steps from the quantizer */
    const void* W8;              /* [K, N] codes of this term's forward weight */
    const float* eps;            /* [T]    from s3r_ec_correct (EC modes 1, 2) */
    const int32_t* rowsum;       /* [K] */
    const float* v;              /* [T/S, K] */
};
int int8_gemm_dx_sum(const struct s3r_dx_term* terms, int n_terms, int code_format, int64_t T, int64_t N, int64_t K,
                     const float* s_x, int ec_mode, int64_t S, float* dX, int accumulate, int* d_status,
                     cudaStream_t stream);

/*
 * int8_gemm_dw -- weight gradient from the same S8 codes ([S3R] §III-A;
 * §III-D weight-gradient term):
 *   acc[k,n] = sum_tb tile_scale[tb, n/128] * (int32) sum_{t in block tb} X8[t,k] Q[t,n]
 *   dW[k,n]  = (acc - sum_b xsum[b,k]*(colmean[b,n] - mu[b]) - p[k]) / s_w[n]  (EC mode 2)
 *   dW[k,n]  = acc / s_w[n]                                                   (EC modes 0, 1)
 * dW is the sum X^T G (not divided by the token count).  S3R_CODES_F16 runs
 * on tcgen05 reading both operands MN-major (needs K % 8 == 0, N % 8 == 0);
 * S3R_CODES_S8 transposes both operands into the workspace first.
 * In : X8 [T, K] codes (the forward input's); Q [T, N] codes; tile_scale;
 *      s_w [N] or NULL; colmean, mu, xsum, p from s3r_ec_correct (mode 2).
 * Out: dW [K, N] fp32 (row stride N).
 * workspace: int8_gemm_dw_workspace_size(T, K, N, code_format) bytes (may be
 * NULL when that is 0).
 */
size_t int8_gemm_dw_workspace_size(int64_t T, int64_t K, int64_t N, int code_format);
int int8_gemm_dw(const void* X8, const void* Q, const float* tile_scale, int code_format, int64_t T, int64_t K,
                 int64_t N, const float* s_w, int ec_mode, const float* colmean, const float* mu,
                 const int32_t* xsum, const float* p, int64_t S, float* dW, void* workspace, size_t workspace_bytes,
                 int* d_status, cudaStream_t stream);

/*
 * int8_gemm_fwd -- the INT8 forward product of one linear ([S3R] §III-A:
 * the forward operands are rounded to nearest with a per-token scale for the
 * input and a per-output-channel scale for the weight, multiplied with S32
 * accumulation and rescaled on both sides):
 *   Y[t, n] = (fp32(acc[t, n]) * s_x[t]) * s_w[n]      in fp32, in this order,
 *   acc     = sum_k X8[t, k] W8[k, n]                   exact (S32; K * 127^2 < 2^31)
 * fp32() rounds to nearest even; only it and the two rescales round.
 * In : X8 [T, K] codes (row stride K), s_x [T]; W8 [K, N] codes as stored
 *      (row stride N), s_w [N].  code_format must be S3R_CODES_F16
 *      (S3R_ERR_UNSUPPORTED otherwise); K and N multiples of 8 and X8, W8
 *      16-byte aligned (S3R_ERR_ALIGN).
 * Out: Y [T, N] fp32 (row stride N).  K == 0 gives Y = 0.
 * One tcgen05 launch; d_status as for int8_gemm_dx.
 */
int int8_gemm_fwd(const void* X8, const float* s_x, const void* W8, const float* s_w, int code_format, int64_t T,
                  int64_t K, int64_t N, float* Y, int* d_status, cudaStream_t stream);

/*
 * int8_gemm_fwd_swiglu -- the gate and up projections of the SwiGLU block
 * (FFN block of [S3R] §IV-A) on one input, with the gate in the epilogue:
 *   h1 = bf16(Y1), h3 = bf16(Y3)     Y1, Y3 as int8_gemm_fwd with (W1_8, s_w1)
 *                                    and (W3_8, s_w3); bf16 = nearest even
 *   a  = bf16((h1 * s) * h3),  s = 1 / (1 + exp(-h1))   in fp32 from the
 *        bf16 h1 and h3, exp as in swiglu_quantize.
 * h1 and h3 are the activations the backward reads; a feeds the next linear.
 * In : X8 [T, K], s_x [T]; W1_8, W3_8 [K, F] (row stride F), s_w1, s_w3 [F];
 *      same format and alignment rules as int8_gemm_fwd.
 * Out: h1, h3 [T, F] bf16 (row stride F); a [T, F] bf16, or NULL to skip the
 *      gate (swiglu_fwd_quantize then forms a together with its codes, the
 *      faster split).  One tcgen05 launch.
 */
int int8_gemm_fwd_swiglu(const void* X8, const float* s_x, const void* W1_8, const float* s_w1, const void* W3_8,
                         const float* s_w3, int code_format, int64_t T, int64_t K, int64_t F, void* h1, void* h3,
                         void* a, int* d_status, cudaStream_t stream);

/*
 * swiglu_fwd_quantize -- the forward SwiGLU gate fused into the per-token
 * RTNE of its output (FFN block of [S3R] §IV-A; §III-A for the operand):
 *   a[t, f] = bf16((h1 * s) * h3),  s = 1 / (1 + exp(-h1))   as in
 *             int8_gemm_fwd_swiglu, from the bf16 h1 and h3;
 *   then Q, scale = rtne_quantize(a, S3R_AXIS_ROW) exactly.
 * In : h1, h3 [T, F] bf16 (row stride ldh).  F and ldh multiples of 8, h1,
 *      h3, a and Q 16-byte aligned (S3R_ERR_ALIGN).
 * Out: a [T, F] bf16 (row stride F) or NULL (not written); Q [T, F] codes in
 *      `code_format`; scale [T].  A row holding a non-finite a gets a NaN
 *      scale, zero codes and *d_status = S3R_ERR_NONFINITE.  One launch.
 */
int swiglu_fwd_quantize(const void* h1, const void* h3, int64_t T, int64_t F, int64_t ldh, void* a, void* Q,
                        int code_format, float* scale, int* d_status, cudaStream_t stream);

/*
 * s3r_sr_bf16 -- stochastic rounding of fp32 to bf16 with S3R's shared
 * thresholds on the hardware stochastic-rounding conversion ([S3R] §II:
 * Blackwell rounds to floating-point formats stochastically from random bits
 * the program supplies; §III-B: one threshold per token).  Per element, on
 * the magnitude: bf16 keeps the upper 16 bits of the fp32 pattern, and moves
 * up one bf16 step iff the 16 dropped bits exceed the 16-bit threshold v
 * (probability = distance to the lower neighbour over the spacing); the sign
 * is kept; beyond the largest finite bf16 (infinities included) saturates to
 * it, NaN becomes 0x7FFF.
 *   round_mode S3R_ROUND_S3R:   v = (w >> 16), w = token t's word as in
 *                               s3r_quantize (Philox4x32-10, counter
 *                               (t mod 2^32, t >> 32, 0, 0), key (seed mod
 *                               2^32, tensor_id)): all channels share it;
 *              S3R_ROUND_INDEP: v = (w_e >> 16), w_e = word (e mod 4) of
 *                               Philox(counter e / 4), e = t N + n;
 *              S3R_ROUND_RTNE:  round to nearest even (no saturation).
 * In : X [T, N] fp32 (row stride ldx).  Out: Y [T, N] bf16 (row stride ldy).
 * 16-byte aligned X, Y with ldx % 4 == 0 and ldy % 8 == 0 take the vector
 * path; any other layout is converted element by element (same results).
 */
int s3r_sr_bf16(const float* X, int64_t T, int64_t N, int64_t ldx, int round_mode, uint64_t seed, uint32_t tensor_id,
                void* Y, int64_t ldy, cudaStream_t stream);

/*
 * s3r_sr_fp8 -- the same rounding to FP8 e4m3 (1 sign, 4 exponent bits with
 * bias 7, 3 mantissa bits; no infinity, largest finite 448), after a scale:
 *   y = x * inv_scale                 fp32, one rounding
 *   e4m3 spacing s = 2^(e-3) for |y| in [2^e, 2^(e+1)), e >= -6, and 2^-9
 *   below 2^-6; with k = floor(|y| / s) and p = |y| / s - k, the magnitude
 *   becomes (k + 1) s iff floor(p 2^16) > v (S3R / INDEP, v as in
 *   s3r_sr_bf16), or rounds to nearest even (RTNE).  The sign is kept;
 *   |y| >= 448 (infinities included) gives +-448, NaN gives 0x7F.
 * In : X [T, N] fp32 (row stride ldx); inv_scale finite and > 0 (S3R_ERR_ARG
 * otherwise: zero, negative, NaN and infinite scales are rejected before any
 * launch).  Out: Y [T, N] e4m3 codes, one byte
 * each (row stride ldy).  16-byte aligned X with ldx % 4 == 0 and 8-byte
 * aligned Y with ldy % 8 == 0 take the vector path; other layouts are
 * converted element by element (same results).
 */
int s3r_sr_fp8(const float* X, int64_t T, int64_t N, int64_t ldx, float inv_scale, int round_mode, uint64_t seed,
               uint32_t tensor_id, void* Y, int64_t ldy, cudaStream_t stream);

/*
 * ffn_forward -- the SwiGLU FFN block forward with INT8 GEMMs, the operands
 * of ffn_backward as its outputs:
 *   1. X8, s_x   = rtne_quantize(X, per row)
 *   2. W1_8, W3_8, W2_8 and their scales = rtne_quantize(W, per column)
 *      (skipped when quantize_weights == 0: they are inputs then)
 *   3. h1, h3    = int8_gemm_fwd_swiglu(X8, W1_8, W3_8)  (a = NULL)
 *   4. a, A8, s_a = swiglu_fwd_quantize(h1, h3)
 *   5. Y         = int8_gemm_fwd(A8, s_a, W2_8, s_w2)
 * All on `stream`, no host synchronization, no workspace.
 */
struct s3r_ffn_fwd_args {
    int64_t T, d, F;             /* tokens, model width, FFN width (d and F multiples of 8) */
    const void* X;               /* bf16 [T, d] */
    const void* W1;              /* bf16 [d, F] (read when quantize_weights) */
    const void* W3;              /* bf16 [d, F] */
    const void* W2;              /* bf16 [F, d] */
    int quantize_weights;        /* 1: step 2 runs; 0: W*_8 and s_w* hold the weights' codes */
    int code_format;             /* S3R_CODES_F16 */
    void* X8;                    /* out [T, d] codes, s_x [T] */
    float* s_x;
    void* W1_8;                  /* out/in [d, F] codes, s_w1 [F] */
    float* s_w1;
    void* W3_8;                  /* out/in [d, F] codes, s_w3 [F] */
    float* s_w3;
    void* W2_8;                  /* out/in [F, d] codes, s_w2 [d] */
    float* s_w2;
    void* h1;                    /* out bf16 [T, F] */
    void* h3;                    /* out bf16 [T, F] */
    void* a;                     /* out bf16 [T, F], or NULL (not kept) */
    void* A8;                    /* out [T, F] codes, s_a [T] */
    float* s_a;
    float* Y;                    /* out fp32 [T, d] */
    int* d_status;               /* device int or NULL */
};
int ffn_forward(const struct s3r_ffn_fwd_args* args, cudaStream_t stream);

/*
 * ffn_backward -- the whole SwiGLU FFN block backward (FFN block of [S3R]
 * §IV-A, Table III), y = (silu(X W1) * (X W3)) W2:
 *   1. quantize dY (fold s_a, s_w2) -> Q2          [tensor id 0]
 *   2. EC factors for W2 (if ec_mode != 0 and round_mode == S3R)
 *   3. dA  = int8_gemm_dx(Q2, W2_8)                [T, F] fp32, in workspace
 *   4. dW2 = int8_gemm_dw(A8, Q2)
 *   5. swiglu_quantize(dA, h1, h3) -> Q1, Q3       [tensor ids 1 (W1), 2 (W3)]
 *   6. EC factors for W1 and W3
 *   7. dX  = int8_gemm_dx_sum({Q1, W1_8}, {Q3, W3_8})
 *   8. dW1 = int8_gemm_dw(X8, Q1), dW3 = int8_gemm_dw(X8, Q3)
 * With fp16 codes, steps 3 and 4 run as one tcgen05 launch and so do steps 7
 * and 8 (each tile computed exactly as in the separate calls); their step
 * events 4 and 8 then follow 3 and 7 directly.
 * Independent SR quantizes each gradient twice (tensor ids + 0x100 for the
 * dW copy) and applies no correction; RTNE applies no correction either.
 *
 * flags & S3R_FFN_FUSE_GLUE (dense block, fp16 codes, round_mode S3R,
 * S3R_7BIT, BCAST or RTNE; ignored otherwise): step 5 runs inside the
 * epilogue of step 3 ([S3R] §III-B: the threshold broadcast and the rounding
 * live inside the fusion that produces the gradient; §IV-A: the SwiGLU
 * block) -- each 128 x 128 tile of dA is turned into dh1 and dh3, folded and
 * quantized where the GEMM holds it, so dA never reaches memory (the
 * workspace's dA is left unwritten).  Q1, Q3 and their tile scales are the
 * same bit for bit as with the separate step 5; the error partials are the
 * same sums in another order.  Step event 5 then follows 4 directly.
 * All buffers are device pointers owned by the caller; `args` itself is a
 * HOST pointer read during the call only.
 *
 * code_format S3R_CODES_S8_F16: X8, A8, W1_8, W3_8 and W2_8 hold int8_t codes
 * (any alignment); the call first copies them, widened to fp16 (exact: every
 * int8 value is an fp16 integer), into the tail of the workspace, then runs
 * the S3R_CODES_F16 block on the copies.  Every result, and every
 * intermediate s3r_ffn_workspace_offsets points at (fp16 codes), equals the
 * S3R_CODES_F16 call on the same codes bit for bit; d and F must be
 * multiples of 8 (S3R_ERR_ALIGN).  The widening runs before the first step
 * event.  The workspace functions take the same
 * code_format and add 2 bytes per operand code (plus alignment) to the
 * S3R_CODES_F16 size.
 *
 * flags & S3R_FFN_RECOMPUTE_A (A8 and s_a NULL, S3R_ERR_ARG otherwise): the
 * call forms the codes of a and their scales itself, from h1 and h3, with the
 * forward's own kernel (swiglu_fwd_quantize: a = bf16(silu(h1) h3), per-token
 * RTNE codes in the format the block computes in), into the tail of the
 * workspace, and then runs the block on them.  The results equal a call
 * given the A8 and s_a that swiglu_fwd_quantize makes from the same h1 and
 * h3, bit for bit; the forward then need not keep A8 (T F codes) at all, and
 * a backward fed from host memory moves that much less.  Workspace:
 * s3r_ffn_workspace_size_flags / s3r_ffn_grouped_workspace_size_flags with
 * the same flags.
 *
 * Grouped (mixture-of-experts) mode, num_groups = E > 0 (the MoE models of
 * [S3R] §IV; the pages give no grouping rule, so the plain one): the T rows
 * of dY, h1, h3, X8/s_x, A8/s_a and dX are routed rows sorted by expert, and
 * expert e owns rows group_offsets[e] .. group_offsets[e+1] (a HOST array of
 * E + 1 non-decreasing offsets, group_offsets[0] = 0, group_offsets[E] = T).
 * The weights are stacked per expert -- W1_8, W3_8 [E, d, F], s_w1, s_w3
 * [E, F], W2_8 [E, F, d], s_w2 [E, d] -- and so are dW1, dW3 [E, d, F] and
 * dW2 [E, F, d].  Each expert runs steps 1-8 on its own rows as one example
 * (S is ignored): tiles and token indices restart at the group's first row
 * and its tensor ids are S3R_MOE_TID_STRIDE * e + (0, 1, 2).  An expert
 * without rows gets zero weight gradients.  Row offsets must keep the bases
 * 16-byte aligned (d and F multiples of 8 for fp16 codes, of 16 for int8).
 * Every step runs for all experts before the next; with fp16 codes each
 * GEMM step is one multi-problem launch over the experts (results equal to
 * per-expert launches bit for bit).  workspace:
 * s3r_ffn_grouped_workspace_size(group_offsets, E, d, F, ...) bytes (one
 * block's buffers per non-empty expert); step events mark the same step
 * boundaries, each over all experts.
 */
#define S3R_TID_W2 0u
#define S3R_TID_W1 1u
#define S3R_TID_W3 2u
#define S3R_TID_RHS_OFFSET 0x100u   /* independent SR: tensor-id offset of the dW copy */
#define S3R_MOE_TID_STRIDE 16u      /* grouped mode: expert e uses ids 16 e + (0, 1, 2) */
struct s3r_ffn_args {
    int64_t T, d, F, S;          /* tokens, model width, FFN width, tokens per example */
    const void* dY;              /* bf16 [T, d] upstream gradient */
    const void* h1;              /* bf16 [T, F] gate pre-activation X W1 */
    const void* h3;              /* bf16 [T, F] up pre-activation X W3 */
    const void* X8;              /* [T, d] RTNE codes of X, per-token scale s_x [T] */
    const float* s_x;
    const void* A8;              /* [T, F] RTNE codes of a = silu(h1)*h3, per-token scale s_a [T] */
    const float* s_a;
    const void* W1_8;            /* [d, F] codes of W1, per-column scale s_w1 [F] */
    const float* s_w1;
    const void* W3_8;            /* [d, F] codes of W3, per-column scale s_w3 [F] */
    const float* s_w3;
    const void* W2_8;            /* [F, d] codes of W2, per-column scale s_w2 [d] */
    const float* s_w2;
    int round_mode;              /* enum s3r_round_mode */
    int ec_mode;                 /* enum s3r_ec_mode (S3R only) */
    int code_format;             /* enum s3r_code_format of the forward codes and of Q1, Q2, Q3 */
    uint64_t seed;
    float* dX;                   /* out [T, d] fp32 */
    float* dW1;                  /* out [d, F] fp32 */
    float* dW3;                  /* out [d, F] fp32 */
    float* dW2;                  /* out [F, d] fp32 */
    void* workspace;
    size_t workspace_bytes;      /* >= s3r_ffn_workspace_size(...) */
    int* d_status;               /* device int or NULL */
    void** step_events;          /* NULL, or S3R_FFN_NUM_EVENTS cudaEvent_t (a HOST array of handles)
                                    recorded on `stream` at the step boundaries: before step 1 and
                                    after steps 1, 2, 3, 4, 5, 6, 7, 8 above (for timing) */
    int64_t num_groups;          /* 0: one dense block; E > 0: grouped mode (above) */
    const int64_t* group_offsets; /* grouped mode: HOST [E + 1] row offsets */
    int flags;                   /* 0, or S3R_FFN_FUSE_GLUE | S3R_FFN_RECOMPUTE_A (above) */
};
#define S3R_FFN_NUM_EVENTS 9
#define S3R_FFN_FUSE_GLUE 1
#define S3R_FFN_RECOMPUTE_A 2
size_t s3r_ffn_workspace_size(int64_t T, int64_t d, int64_t F, int64_t S, int round_mode, int ec_mode,
                              int code_format);
/* grouped mode: group_offsets is the HOST [num_groups + 1] array of the call;
   0 for invalid offsets */
size_t s3r_ffn_grouped_workspace_size(const int64_t* group_offsets, int64_t num_groups, int64_t d, int64_t F,
                                      int round_mode, int ec_mode, int code_format);
/* the workspace of a call with these flags (S3R_FFN_RECOMPUTE_A adds the
   recomputed codes of a and their scales); 0 for invalid sizes */
size_t s3r_ffn_workspace_size_flags(int64_t T, int64_t d, int64_t F, int64_t S, int round_mode, int ec_mode,
                                    int code_format, int flags);
size_t s3r_ffn_grouped_workspace_size_flags(const int64_t* group_offsets, int64_t num_groups, int64_t d, int64_t F,
                                            int round_mode, int ec_mode, int code_format, int flags);
int ffn_backward(const struct s3r_ffn_args* args, cudaStream_t stream);

/*
 * s3r_ffn_workspace_offsets -- inspection hook: where ffn_backward keeps its
 * intermediates inside the caller's workspace, so that a test can compare
 * them with a reference after the call.  Writes to `out` (a HOST array of
 * S3R_FFN_WS_VIEWS entries) the byte offsets, from a workspace base aligned
 * to 256 bytes, of
 *   [0] Q2 codes [T, d]   [1] Q2 tile scales [ceil(T/128), ceil(d/128)]
 *   [2] Q1 codes [T, F]   [3] Q1 tile scales [ceil(T/128), ceil(F/128)]
 *   [4] Q3 codes [T, F]   [5] Q3 tile scales
 *   [6] dA [T, F] fp32 (the activation gradient of W2, input of the glue)
 * codes in `code_format` (fp16 for S3R_CODES_S8_F16, whose block runs on
 * fp16 codes), all row-major with the listed widths.  num_groups
 * = 0: the dense block (T, S as in ffn_backward).  num_groups = E > 0: the
 * block of expert `group` (0 <= group < E) under the HOST group_offsets of
 * the grouped call (T and S ignored; the shapes use the group's row count).
 * S3R_ERR_ARG for invalid sizes, an empty group or a NULL `out`.
 * Host-only: launches nothing.
 */
#define S3R_FFN_WS_VIEWS 7
int s3r_ffn_workspace_offsets(int64_t T, int64_t d, int64_t F, int64_t S, int round_mode, int code_format,
                              const int64_t* group_offsets, int64_t num_groups, int64_t group, size_t* out);

/*
 * Test hooks: the exact int32 per-block partial products computed by the
 * same tensor-core main loops as int8_gemm_dx / int8_gemm_dw, before any
 * rescale.  out_dx [T, K, ceil(N/128)]: block kb of sum_n Q[t,n] W8[k,n];
 * out_dw [K, N, ceil(T/128)]: block tb of sum_t X8[t,k] Q[t,n].  int32.
 */
int s3r_debug_dx_blocks(const void* Q, const void* W8, int code_format, int64_t T, int64_t N, int64_t K,
                        int32_t* out_dx, cudaStream_t stream);
int s3r_debug_dw_blocks(const void* X8, const void* Q, int code_format, int64_t T, int64_t K, int64_t N,
                        int32_t* out_dw, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Test hook for the reciprocal inside the SwiGLU glue (sigma = 1 / (1 + e)
 * of the SwiGLU block, [S3R] section IV-A), which must equal the IEEE
 * quotient bit for bit so that the codes downstream of the glue match an
 * implementation that divides: counts the floats
 * whose bit patterns lie in [lo_bits, hi_bits) (positive, finite, lo_bits <
 * hi_bits <= 0x7F800000) for which the kernels' reciprocal differs from the
 * correctly rounded IEEE reciprocal, adding the count into *d_count (device
 * memory, caller-owned, one unsigned 64-bit integer).  Asynchronous on
 * `stream`.  S3R_ERR_ARG for an invalid range or a NULL d_count.
 */
int s3r_check_reciprocal(uint32_t lo_bits, uint32_t hi_bits, unsigned long long* d_count, cudaStream_t stream);

/*
 * Test hook for failure detection (no counterpart on the pages): every wait
 * inside the kernels is bounded -- it gives up after its limit (2 s) or, where
 * the kernel has one, as soon as another role of the CTA raised its abort
 * flag -- and a kernel whose wait gave up writes S3R_ERR_TIMEOUT to d_status
 * and exits cleanly, leaving the context usable.  This runs the wait routine
 * of one kernel family (family: S3R_WAIT_GEMM, S3R_WAIT_QUANTIZE or
 * S3R_WAIT_EC) in a one-CTA launch on an mbarrier that nothing arrives on,
 * with the limit limit_ns (0 < limit_ns <= 2e9); raise_abort != 0 (GEMM and
 * EC families only) has a second warp raise the abort flag after about 1 ms
 * instead.  The waiter writes the nanoseconds it waited to *d_waited_ns and
 * S3R_ERR_TIMEOUT to *d_status (both device memory).  Asynchronous on `stream`.
 * S3R_ERR_ARG for a bad family, limit or pointer.
 */
#define S3R_WAIT_GEMM 0
#define S3R_WAIT_QUANTIZE 1
#define S3R_WAIT_EC 2
int s3r_debug_wait_timeout(int family, uint64_t limit_ns, int raise_abort, int* d_status,
                           unsigned long long* d_waited_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* S3R_H */
