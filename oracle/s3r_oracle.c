/*
 * s3r_oracle.c -- plain, single-threaded CPU oracle for the S3R / S3R-EC INT8
 * backward.  TEST INFRASTRUCTURE ONLY: the product path never links, loads or
 * calls this file; only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or constant generator
 * with the CUDA library.
 *
 * Sources (cited by page title and section):
 *   [S3R]  "Efficient Quantization Training with Stochastic Rounding via
 *          Structured Subspace Randomness" (sections rebuilt from the text:
 *          §III-A quantized backprop with SR, §III-B structured subspace
 *          randomness, §III-C why sharing hurts, §III-D S3R-EC, §IV-B compared
 *          configurations).
 *   [SRB]  "Stochastic Rounding" (transformer-math blog): sections "Stochastic
 *          rounding, defined", "The probability formula".
 *   [PHX]  Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
 *          1, 2, 3", SC'11: the Philox4x32-10 bijection (cited by [S3R] §II).
 *
 * Precision.  Where floating point decides an integer code (fold, tile scale,
 * normalised value, residual, threshold compare) this file uses exactly the
 * fp32 operations the kernels use, in the order stated below, so codes can be
 * compared bit for bit.  Reductions, error statistics, correction factors and
 * the GEMM rescale are computed in fp64.  Compile with -ffp-contract=off so no
 * multiply-add is fused behind our back.
 *
 * Nothing here is blocked, fused or reordered beyond the definitions: every
 * function is a direct loop over the formula it cites.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG (-1)
#define ORC_ERR_NONFINITE (-4)

/* rounding modes */
#define ORC_RTNE 0
#define ORC_S3R 1   /* one threshold per token, shared by its channels (Phi_2D) */
#define ORC_INDEP 2 /* one threshold per element */
#define ORC_S3R7 3  /* Phi_2D with 7-bit thresholds, four per word, shifted by half a step */
#define ORC_BCAST 4 /* one threshold per example, shared by all its tokens and channels (Phi_bcast) */

/* error-correction modes */
#define ORC_EC_NONE 0
#define ORC_EC_DX_ONLY 1     /* full activation-gradient term of the projection */
#define ORC_EC_TWO_WAY 2     /* both products */
#define ORC_EC_DX_TOKEN_ONLY 3 /* alternative reading: token-mean term eps*r only */
#define ORC_EC_DW_ONLY 4     /* ablation: the weight-gradient term only */

/* ------------------------------------------------------------------------- */
/* Philox4x32-10 [PHX]: 10 rounds of the Philox S-box on a 4x32-bit counter   */
/* with a 2x32-bit key bumped by the Weyl constants between rounds.           */
/* ------------------------------------------------------------------------- */
void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u; /* golden ratio */
            k1 += 0xBB67AE85u; /* sqrt(3) - 1 */
        }
        uint64_t prod0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t prod1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* A 32-bit word to a threshold on the 24-bit grid in [0, 1): (w >> 8) * 2^-24. */
float orc_word_to_unit(uint32_t w) {
    return (float)(w >> 8) * 0x1.0p-24f;
}

/* [S3R] §III-B "Threshold broadcasting", Phi_2D: one uniform threshold u_t per
 * token, shared by all channels of that token.  Counter = token index t,
 * key = (low 32 bits of seed, tensor id); the threshold is output word 0. */
float orc_token_threshold(uint64_t t, uint64_t seed, uint32_t tensor_id) {
    uint32_t ctr[4] = {(uint32_t)t, (uint32_t)(t >> 32), 0u, 0u};
    uint32_t key[2] = {(uint32_t)seed, tensor_id};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    return orc_word_to_unit(out[0]);
}

/* [S3R] §III-B "Structured subspace randomness": the paper's own thresholds
 * are 7-bit values, four cut from each 32-bit word, on a grid shifted by half
 * a step.  Token t takes byte (t mod 4) of output word 0 of Philox(counter =
 * t / 4); of that byte the upper 7 bits k give u = (k + 1/2) / 128, so u takes
 * the 128 values 1/256, 3/256, ..., 255/256 and P(u < p) differs from p by at
 * most 1/256 (the pages' bound Delta/256 on the bias). */
float orc_token_threshold7(uint64_t t, uint64_t seed, uint32_t tensor_id) {
    uint64_t c = t >> 2;
    uint32_t ctr[4] = {(uint32_t)c, (uint32_t)(c >> 32), 0u, 0u};
    uint32_t key[2] = {(uint32_t)seed, tensor_id};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    uint32_t byte = (out[0] >> (8u * (uint32_t)(t & 3u))) & 0xFFu;
    return ((float)(byte >> 1) + 0.5f) / 128.0f;
}

/* [S3R] §III-B, Phi_bcast (the ablation): one threshold u_b per example b,
 * shared by all its tokens and channels.  Counter = (b, 0, 1, 0) (counter
 * word 2 = 1 keeps these draws apart from the per-token ones), same key and
 * 24-bit grid as Phi_2D. */
float orc_example_threshold(uint64_t b, uint64_t seed, uint32_t tensor_id) {
    uint32_t ctr[4] = {(uint32_t)b, (uint32_t)(b >> 32), 1u, 0u};
    uint32_t key[2] = {(uint32_t)seed, tensor_id};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    return orc_word_to_unit(out[0]);
}

/* [S3R] §III-A, conventional QT: an independent threshold for every element.
 * Element e = t*N + n uses word (e mod 4) of Philox(counter = e / 4). */
float orc_element_threshold(uint64_t e, uint64_t seed, uint32_t tensor_id) {
    uint64_t c = e >> 2;
    uint32_t ctr[4] = {(uint32_t)c, (uint32_t)(c >> 32), 0u, 0u};
    uint32_t key[2] = {(uint32_t)seed, tensor_id};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    return orc_word_to_unit(out[e & 3]);
}

/* bf16 bit pattern to fp32 (exact). */
float orc_bf16_to_float(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

void orc_bf16_array_to_float(const uint16_t* src, int64_t n, float* dst) {
    for (int64_t i = 0; i < n; ++i) dst[i] = orc_bf16_to_float(src[i]);
}

/* ------------------------------------------------------------------------- */
/* Quantization of the backward gradient ([S3R] §III-A).                      */
/*                                                                            */
/* For each element, in fp32:                                                 */
/*   fold      g  = (s_x[t] * G[t,n]) * s_w[n]      (null scale pointer = 1)  */
/*   scale     amax = max |g| over the tile; delta = amax / 127 (nearest);    */
/*             inv = 127 / amax rounded toward zero, so |g * inv| <= 127     */
/*             and no code leaves [-127, 127] (delta = inv = 0 if amax == 0) */
/*   normalise y  = g * inv                                                   */
/*   SR        f = floor(y); p = y - f; q = f + [u < p]   ([SRB] "u < p")     */
/*   RTNE      q = nearbyint(y)  (round half to even)                         */
/*   clamp     q in [-127, 127]                                               */
/*   error     e = fma(delta, q, -g)     (E = delta*Q - G', [S3R] §III-A)     */
/* Tiles are tr x tc and start at row 0 / column 0; the last ones may be      */
/* partial.  delta is [ceil(T/tr), ceil(N/tc)] row-major.  E may be NULL.     */
/* ------------------------------------------------------------------------- */
/* The scalar SR step on a grid of unit spacing ([SRB] "Stochastic rounding,
 * defined" / "The probability formula"; [S3R] §III-A): with f = floor(y) and
 * residual p = y - f, round up to f + 1 when the threshold u lies below p,
 * otherwise down to f.  A value on the grid (p = 0) never moves. */
float orc_sr_step(float y, float u) {
    float f = floorf(y);
    float p = y - f;
    return (u < p) ? f + 1.0f : f;
}

/* 127 / a rounded toward zero (a > 0): the nearest quotient, stepped down
 * one ulp when it overshoots (the fma residual 127 - q*a is exact in sign). */
float orc_inv127_rz(float a) {
    float q = 127.0f / a;
    if (fmaf(-q, a, 127.0f) < 0.0f) q = nextafterf(q, 0.0f);
    return q;
}

static float fold_one(const float* G, int64_t ldg, const float* s_x, const float* s_w, int64_t t, int64_t n) {
    float g = G[t * ldg + n];
    if (s_x) g = s_x[t] * g;
    if (s_w) g = g * s_w[n];
    return g;
}

/* orc_quantize_window: the same on a tile-aligned window of a larger tensor
 * whose first row is global token row_base and first column is col_base, in a
 * tensor of n_global columns; only the threshold indices use these (token
 * t + row_base; element (t + row_base) * n_global + col_base + n). */
/* S is the number of tokens per example (Phi_bcast: example of token t is
 * t / S; S <= 0 means one example). */
int orc_quantize_window_ex(const float* G, int64_t T, int64_t N, int64_t ldg,
                           const float* s_x, const float* s_w, int mode, int64_t S, uint64_t seed,
                           uint32_t tensor_id, int64_t tr, int64_t tc, int8_t* Q, float* delta, float* E,
                           int64_t row_base, int64_t col_base, int64_t n_global) {
    if (T < 0 || N < 0 || tr <= 0 || tc <= 0 || ldg < N) return ORC_ERR_ARG;
    if (mode != ORC_RTNE && mode != ORC_S3R && mode != ORC_INDEP && mode != ORC_S3R7 && mode != ORC_BCAST)
        return ORC_ERR_ARG;
    int status = ORC_OK;
    int64_t ntr = (T + tr - 1) / tr, ntc = (N + tc - 1) / tc;
    for (int64_t i = 0; i < ntr; ++i) {
        for (int64_t j = 0; j < ntc; ++j) {
            int64_t t0 = i * tr, t1 = (t0 + tr < T) ? t0 + tr : T;
            int64_t n0 = j * tc, n1 = (n0 + tc < N) ? n0 + tc : N;
            /* tile absmax of the folded gradient */
            float amax = 0.0f;
            int finite = 1;
            for (int64_t t = t0; t < t1; ++t)
                for (int64_t n = n0; n < n1; ++n) {
                    float g = fold_one(G, ldg, s_x, s_w, t, n);
                    if (!isfinite(g)) finite = 0;
                    else if (fabsf(g) > amax) amax = fabsf(g);
                }
            if (!finite) {
                status = ORC_ERR_NONFINITE;
                delta[i * ntc + j] = NAN;
                for (int64_t t = t0; t < t1; ++t)
                    for (int64_t n = n0; n < n1; ++n) {
                        Q[t * N + n] = 0;
                        if (E) E[t * N + n] = 0.0f;
                    }
                continue;
            }
            float d = amax / 127.0f;
            float inv = (amax > 0.0f) ? orc_inv127_rz(amax) : 0.0f;
            delta[i * ntc + j] = d;
            for (int64_t t = t0; t < t1; ++t) {
                const uint64_t tg = (uint64_t)(t + row_base);
                float u_tok = 0.0f;
                if (mode == ORC_S3R) u_tok = orc_token_threshold(tg, seed, tensor_id);
                else if (mode == ORC_S3R7) u_tok = orc_token_threshold7(tg, seed, tensor_id);
                else if (mode == ORC_BCAST) u_tok = orc_example_threshold(S > 0 ? tg / (uint64_t)S : 0u, seed, tensor_id);
                for (int64_t n = n0; n < n1; ++n) {
                    float g = fold_one(G, ldg, s_x, s_w, t, n);
                    float y = g * inv;
                    float qf;
                    if (mode == ORC_RTNE) {
                        qf = nearbyintf(y);
                    } else {
                        float u = (mode != ORC_INDEP)
                                      ? u_tok
                                      : orc_element_threshold((uint64_t)((t + row_base) * n_global + col_base + n),
                                                              seed, tensor_id);
                        qf = orc_sr_step(y, u);
                    }
                    if (qf > 127.0f) qf = 127.0f;
                    if (qf < -127.0f) qf = -127.0f;
                    Q[t * N + n] = (int8_t)qf;
                    if (E) E[t * N + n] = fmaf(d, qf, -g);
                }
            }
        }
    }
    return status;
}

int orc_quantize_window(const float* G, int64_t T, int64_t N, int64_t ldg,
                        const float* s_x, const float* s_w, int mode, uint64_t seed, uint32_t tensor_id,
                        int64_t tr, int64_t tc, int8_t* Q, float* delta, float* E,
                        int64_t row_base, int64_t col_base, int64_t n_global) {
    return orc_quantize_window_ex(G, T, N, ldg, s_x, s_w, mode, 0, seed, tensor_id, tr, tc, Q, delta, E, row_base,
                                  col_base, n_global);
}

int orc_quantize(const float* G, int64_t T, int64_t N, int64_t ldg,
                 const float* s_x, const float* s_w, int mode, uint64_t seed, uint32_t tensor_id,
                 int64_t tr, int64_t tc, int8_t* Q, float* delta, float* E) {
    return orc_quantize_window(G, T, N, ldg, s_x, s_w, mode, seed, tensor_id, tr, tc, Q, delta, E, 0, 0, N);
}

/* Forward operands ([S3R] §III-A): RTNE with a per-row (axis 0) or per-column
 * (axis 1) absmax scale s = amax/127, so that A ~= diag(s) A_hat (rows) or
 * A ~= A_hat diag(s) (columns).  An all-zero row/column gets s = 1: any scale
 * reproduces zero, and 1 keeps the backward fold and rescale finite. */
int orc_rtne_operand(const float* A, int64_t R, int64_t C, int64_t lda, int axis, int8_t* Q, float* scale) {
    if (R < 0 || C < 0 || lda < C || (axis != 0 && axis != 1)) return ORC_ERR_ARG;
    int64_t nvec = axis == 0 ? R : C, len = axis == 0 ? C : R;
    for (int64_t v = 0; v < nvec; ++v) {
        float amax = 0.0f;
        for (int64_t l = 0; l < len; ++l) {
            float a = axis == 0 ? A[v * lda + l] : A[l * lda + v];
            if (!isfinite(a)) return ORC_ERR_NONFINITE;
            if (fabsf(a) > amax) amax = fabsf(a);
        }
        float s = amax > 0.0f ? amax / 127.0f : 1.0f;
        float inv = amax > 0.0f ? orc_inv127_rz(amax) : 1.0f;
        scale[v] = s;
        for (int64_t l = 0; l < len; ++l) {
            int64_t r = axis == 0 ? v : l, c = axis == 0 ? l : v;
            float qf = nearbyintf(A[r * lda + c] * inv);
            if (qf > 127.0f) qf = 127.0f;
            if (qf < -127.0f) qf = -127.0f;
            Q[r * C + c] = (int8_t)qf;
        }
    }
    return ORC_OK;
}

/* Per-tile partial sums of the rounding error, the quantities the quantizer
 * hands to the correction: tok[t, j] = sum over tile column j of e[t, n];
 * col[i, n] = sum over tile row i of e[t, n]. */
void orc_error_partials(const float* E, int64_t T, int64_t N, int64_t tr, int64_t tc, double* tok, double* col) {
    int64_t ntr = (T + tr - 1) / tr, ntc = (N + tc - 1) / tc;
    for (int64_t i = 0; i < T * ntc; ++i) tok[i] = 0.0;
    for (int64_t i = 0; i < ntr * N; ++i) col[i] = 0.0;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t n = 0; n < N; ++n) {
            tok[t * ntc + n / tc] += (double)E[t * N + n];
            col[(t / tr) * N + n] += (double)E[t * N + n];
        }
}

/* [S3R] §III-D "Two-way correction": the averages of the rounding error of
 * example b (S consecutive tokens, T = B*S): token means eps[t] over the N
 * channels, channel means colmean[b, n] over the S tokens, and the grand
 * mean mu[b].  Together they give the orthogonal projection of E_b onto
 * {1_S a^T + c 1_D^T}: P(E_b) = 1_S colmean_b^T + eps_b 1_D^T - mu_b 1 1^T. */
int orc_error_stats(const float* E, int64_t T, int64_t N, int64_t S, double* eps, double* colmean, double* mu) {
    if (S <= 0 || T % S != 0) return ORC_ERR_ARG;
    int64_t B = T / S;
    for (int64_t t = 0; t < T; ++t) {
        double s = 0.0;
        for (int64_t n = 0; n < N; ++n) s += (double)E[t * N + n];
        eps[t] = s / (double)N;
    }
    for (int64_t b = 0; b < B; ++b) {
        double total = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0;
            for (int64_t t = b * S; t < (b + 1) * S; ++t) s += (double)E[t * N + n];
            colmean[b * N + n] = s / (double)S;
            total += s;
        }
        mu[b] = total / ((double)S * (double)N);
    }
    return ORC_OK;
}

/* [S3R] §III-D: the factors through which P(E) enters the two products.
 *   rowsum[k]  = sum_n W8[k, n]                (W 1_D, "precomputed row sums")
 *   v[b, k]    = sum_n (colmean[b,n] - mu[b]) W8[k, n]
 *   xsum[b, k] = sum_{t in b} X8[t, k]          (= S * xbar_b)
 *   p[k]       = sum_t X8[t, k] eps[t]
 * so that  P(E_b) W8^T [t, k] = eps[t] rowsum[k] + v[b, k]  and
 *          X8^T P(E) [k, n]   = sum_b xsum[b,k] (colmean[b,n] - mu[b]) + p[k].
 * W8 is [K, N] (the weight of Y = X W with K = H_in, N = H_out), X8 is [T, K].
 * X8 may be NULL (then xsum and p are not written). */
void orc_ec_factors(const double* eps, const double* colmean, const double* mu,
                    int64_t T, int64_t N, int64_t S, const int8_t* W8, const int8_t* X8, int64_t K,
                    int64_t* rowsum, double* v, int64_t* xsum, double* p) {
    int64_t B = T / S;
    for (int64_t k = 0; k < K; ++k) {
        int64_t r = 0;
        for (int64_t n = 0; n < N; ++n) r += W8[k * N + n];
        rowsum[k] = r;
        for (int64_t b = 0; b < B; ++b) {
            double s = 0.0;
            for (int64_t n = 0; n < N; ++n) s += (colmean[b * N + n] - mu[b]) * (double)W8[k * N + n];
            v[b * K + k] = s;
        }
    }
    if (!X8) return;
    for (int64_t k = 0; k < K; ++k) {
        double pk = 0.0;
        for (int64_t b = 0; b < B; ++b) {
            int64_t s = 0;
            for (int64_t t = b * S; t < (b + 1) * S; ++t) s += X8[t * K + k];
            xsum[b * K + k] = s;
        }
        for (int64_t t = 0; t < T; ++t) pk += (double)X8[t * K + k] * eps[t];
        p[k] = pk;
    }
}

/* Exact integer partial products per 128-wide contraction block (the S8 GEMM
 * with S32 accumulation of [S3R] §III-A), straight from the definition.
 *   dX block kb: I[r, k, kb] = sum_{n in block kb} Q[t_r, n] W8[k, n]
 *   dW block tb: J[r, n, tb] = sum_{t in block tb} X8[t, k_r] Q[t, n]
 * Only the requested rows (t_r for dX, k_r for dW) are produced. */
void orc_dx_blocks(const int8_t* Q, const int8_t* W8, int64_t T, int64_t N, int64_t K, int64_t blk,
                   const int64_t* rows, int64_t nrows, int32_t* I) {
    int64_t nkb = (N + blk - 1) / blk;
    (void)T;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t t = rows[r];
        for (int64_t k = 0; k < K; ++k)
            for (int64_t kb = 0; kb < nkb; ++kb) {
                int64_t s = 0;
                for (int64_t n = kb * blk; n < N && n < (kb + 1) * blk; ++n) s += (int64_t)Q[t * N + n] * W8[k * N + n];
                I[(r * K + k) * nkb + kb] = (int32_t)s;
            }
    }
}

void orc_dw_blocks(const int8_t* X8, const int8_t* Q, int64_t T, int64_t K, int64_t N, int64_t blk,
                   const int64_t* krows, int64_t nk, int32_t* J) {
    int64_t ntb = (T + blk - 1) / blk;
    int64_t* acc = (int64_t*)malloc(sizeof(int64_t) * (size_t)(N > 0 ? N : 1));
    for (int64_t r = 0; r < nk; ++r) {
        int64_t k = krows[r];
        for (int64_t tb = 0; tb < ntb; ++tb) {
            /* integer sums: the order of the t loop does not change them */
            for (int64_t n = 0; n < N; ++n) acc[n] = 0;
            for (int64_t t = tb * blk; t < T && t < (tb + 1) * blk; ++t) {
                int64_t x = X8[t * K + k];
                for (int64_t n = 0; n < N; ++n) acc[n] += x * Q[t * N + n];
            }
            for (int64_t n = 0; n < N; ++n) J[(r * N + n) * ntb + tb] = (int32_t)acc[n];
        }
    }
    free(acc);
}

/* Activation gradient ([S3R] §III-A, §III-D), for the requested token rows:
 *   acc[t,k] = sum_kb delta[t/tr, kb] * I[t, k, kb]          (rescale, fp64)
 *   corr     = eps[t] rowsum[k] + v[b(t), k]    (EC_DX_ONLY, EC_TWO_WAY)
 *            = eps[t] rowsum[k]                 (EC_DX_TOKEN_ONLY)
 *   dX[t,k]  = (acc - corr) / s_x[t]            (s_x NULL = 1)
 * The contraction blocks are the tile columns of Q (blk = tc). */
void orc_dx(const int8_t* Q, const float* delta, const int8_t* W8, int64_t T, int64_t N, int64_t K,
            int64_t tr, int64_t tc, const float* s_x, int ec_mode, const double* eps, const int64_t* rowsum,
            const double* v, int64_t S, const int64_t* rows, int64_t nrows, double* dX) {
    int64_t nkb = (N + tc - 1) / tc;
    int32_t* I = (int32_t*)malloc(sizeof(int32_t) * (size_t)(K * nkb > 0 ? K * nkb : 1));
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t t = rows[r];
        orc_dx_blocks(Q, W8, T, N, K, tc, &t, 1, I);
        for (int64_t k = 0; k < K; ++k) {
            double acc = 0.0;
            for (int64_t kb = 0; kb < nkb; ++kb) acc += (double)delta[(t / tr) * nkb + kb] * (double)I[k * nkb + kb];
            double corr = 0.0;
            if (ec_mode == ORC_EC_DX_ONLY || ec_mode == ORC_EC_TWO_WAY)
                corr = eps[t] * (double)rowsum[k] + v[(t / S) * K + k];
            else if (ec_mode == ORC_EC_DX_TOKEN_ONLY)
                corr = eps[t] * (double)rowsum[k];
            double sx = s_x ? (double)s_x[t] : 1.0;
            dX[r * K + k] = (acc - corr) / sx;
        }
    }
    free(I);
}

/* Weight gradient ([S3R] §III-A, §III-D), for the requested rows k of dW [K, N]:
 *   acc[k,n] = sum_tb delta[tb, n/tc] * J[k, n, tb]
 *   corr     = sum_b xsum[b,k] (colmean[b,n] - mu[b]) + p[k]   (EC_TWO_WAY, EC_DW_ONLY)
 *   dW[k,n]  = (acc - corr) / s_w[n]                            (s_w NULL = 1)
 * The contraction blocks are the tile rows of Q (blk = tr).  dW is the sum
 * X^T G, not divided by the token count ([S3R] §III-A leaves 1/(BS) to the
 * caller). */
void orc_dw(const int8_t* X8, const int8_t* Q, const float* delta, int64_t T, int64_t K, int64_t N,
            int64_t tr, int64_t tc, const float* s_w, int ec_mode, const double* colmean, const double* mu,
            const int64_t* xsum, const double* p, int64_t S, const int64_t* krows, int64_t nk, double* dW) {
    int64_t ntb = (T + tr - 1) / tr, ntc = (N + tc - 1) / tc, B = T / S;
    int32_t* J = (int32_t*)malloc(sizeof(int32_t) * (size_t)(N * ntb > 0 ? N * ntb : 1));
    for (int64_t r = 0; r < nk; ++r) {
        int64_t k = krows[r];
        orc_dw_blocks(X8, Q, T, K, N, tr, &k, 1, J);
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t tb = 0; tb < ntb; ++tb) acc += (double)delta[tb * ntc + n / tc] * (double)J[n * ntb + tb];
            double corr = 0.0;
            if (ec_mode == ORC_EC_TWO_WAY || ec_mode == ORC_EC_DW_ONLY) {
                for (int64_t b = 0; b < B; ++b) corr += (double)xsum[b * K + k] * (colmean[b * N + n] - mu[b]);
                corr += p[k];
            }
            double sw = s_w ? (double)s_w[n] : 1.0;
            dW[r * N + n] = (acc - corr) / sw;
        }
    }
    free(J);
}

/* ------------------------------------------------------------------------- */
/* SwiGLU backward glue (the FFN block of [S3R] §IV-A / Table III).           */
/* exp: Cody-Waite argument reduction x = n ln2 + r with ln2 split in a       */
/* 16-bit head and a tail, |r| <= ln2/2, e^r by its degree-7 Taylor series in */
/* Horner form, then scaling by 2^n.  The argument is clamped to [-87, 88] so */
/* 2^n stays a normal number.                                                 */
/* ------------------------------------------------------------------------- */
float orc_expf(float x) {
    if (x > 88.0f) x = 88.0f;
    if (x < -87.0f) x = -87.0f;
    const float log2e = 0x1.715476p+0f;     /* log2(e) rounded to fp32 */
    const float ln2_hi = 0x1.62e4p-1f;      /* 45426 / 2^16 */
    const float ln2_lo = 0x1.7f7d1cp-20f;   /* ln2 - ln2_hi rounded to fp32 */
    float n = nearbyintf(x * log2e);
    float r = fmaf(-n, ln2_hi, x);
    r = fmaf(-n, ln2_lo, r);
    float poly = 0x1.a01a02p-13f;           /* 1/7! */
    poly = fmaf(poly, r, 0x1.6c16c2p-10f);  /* 1/6! */
    poly = fmaf(poly, r, 0x1.111112p-7f);   /* 1/5! */
    poly = fmaf(poly, r, 0x1.555556p-5f);   /* 1/4! */
    poly = fmaf(poly, r, 0x1.555556p-3f);   /* 1/3! */
    poly = fmaf(poly, r, 0.5f);             /* 1/2! */
    poly = fmaf(poly, r, 1.0f);
    poly = fmaf(poly, r, 1.0f);
    int32_t ni = (int32_t)n;
    uint32_t bits = (uint32_t)(ni + 127) << 23;
    float scale;
    memcpy(&scale, &bits, 4);
    return poly * scale;
}

float orc_sigmoidf(float x) {
    float e = orc_expf(-x);
    return 1.0f / (1.0f + e);
}

/* With a = silu(h1) * h3 and dA = dL/da (fp32), in fp32 and in this order:
 *   s    = sigmoid(h1)
 *   silu = h1 * s
 *   dsilu = s * (1 + h1 * (1 - s))        (d silu / d h1)
 *   dh1  = (dA * h3) * dsilu
 *   dh3  = dA * silu                                                          */
void orc_swiglu_bwd(const float* dA, const float* h1, const float* h3, int64_t n, float* dh1, float* dh3) {
    for (int64_t i = 0; i < n; ++i) {
        float s = orc_sigmoidf(h1[i]);
        float silu = h1[i] * s;
        float one_minus = 1.0f - s;
        float inner = h1[i] * one_minus;
        float dsilu = s * (1.0f + inner);
        float g = dA[i] * h3[i];
        dh1[i] = g * dsilu;
        dh3[i] = dA[i] * silu;
    }
}

/* ------------------------------------------------------------------------- */
/* INT8 forward ([S3R] §III-A: Y = diag(s_x) X_hat W_hat diag(s_w), with the  */
/* RTNE operands of orc_rtne_operand).  S8 x S8 products accumulate exactly  */
/* as integers (the section's S32 accumulation), the sum is converted to fp32 */
/* once (round to nearest even) and rescaled in fp32 as (acc * s_x[t]) *      */
/* s_w[n].  X8 [T, K] int8, W8 [K, N] int8, Y [T, N] fp32.                    */
/* ------------------------------------------------------------------------- */
void orc_gemm_fwd(const int8_t* X8, const float* s_x, const int8_t* W8, const float* s_w, int64_t T, int64_t K,
                  int64_t N, float* Y) {
    for (int64_t t = 0; t < T; ++t)
        for (int64_t n = 0; n < N; ++n) {
            int64_t acc = 0;
            for (int64_t k = 0; k < K; ++k) acc += (int64_t)X8[t * K + k] * (int64_t)W8[k * N + n];
            float y = (float)acc * s_x[t];
            Y[t * N + n] = y * s_w[n];
        }
}

/* fp32 to bf16 bits, rounded to nearest even (NaN kept quiet). */
uint16_t orc_float_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* The SwiGLU gate of the forward (the FFN block of [S3R] §IV-A): the GEMM
 * outputs are saved as bf16 (h1, h3: the activations the backward reads), and
 * a = silu(h1) * h3 is formed from those bf16 values in fp32, in this order:
 *   s = sigmoid(h1),  silu = h1 * s,  a = bf16(silu * h3). */
void orc_swiglu_fwd(const float* h1f, const float* h3f, int64_t n, uint16_t* h1b, uint16_t* h3b, uint16_t* ab) {
    for (int64_t i = 0; i < n; ++i) {
        h1b[i] = orc_float_to_bf16(h1f[i]);
        h3b[i] = orc_float_to_bf16(h3f[i]);
        float x = orc_bf16_to_float(h1b[i]), z = orc_bf16_to_float(h3b[i]);
        float s = orc_sigmoidf(x);
        float silu = x * s;
        ab[i] = orc_float_to_bf16(silu * z);
    }
}

/* ------------------------------------------------------------------------- */
/* Stochastic rounding of fp32 to bf16 with 16-bit thresholds.  [S3R] §II:   */
/* the hardware conversion to floating-point formats rounds stochastically    */
/* from random bits the program supplies; §III-B: one threshold per token,    */
/* shared by all its channels.  On the magnitude: bf16 keeps the upper 16     */
/* bits of the fp32 pattern.  With L the 16 dropped bits and v a 16-bit       */
/* threshold, the magnitude moves up one bf16 step iff L > v; for v uniform   */
/* on 0..65535 that has probability L / 2^16, the distance to the lower       */
/* neighbour over the spacing ([SRB] "The probability formula").  Values      */
/* beyond the largest finite bf16 (infinities included) saturate to it, NaN   */
/* becomes 0x7FFF: the saturating rule of the conversion the kernels use.     */
/* ------------------------------------------------------------------------- */
uint16_t orc_sr_bf16(float x, uint32_t v) {
    uint32_t u;
    memcpy(&u, &x, 4);
    uint32_t sign = (u >> 16) & 0x8000u, mag = u & 0x7FFFFFFFu;
    if (mag > 0x7F800000u) return 0x7FFFu;
    uint32_t hi = mag >> 16, low = mag & 0xFFFFu;
    if (low > (v & 0xFFFFu)) hi += 1u;
    if (hi >= 0x7F80u) hi = 0x7F7Fu;
    return (uint16_t)(sign | hi);
}

/* X [T, N] fp32 (row stride ldx) -> Y [T, N] bf16 bits (row stride N); row i
 * is token t = t0 + i (t0 > 0 evaluates a window of a larger tensor).
 *   ORC_S3R:   v = the upper 16 bits of token t's word (word 0 of
 *              Philox(counter = (t, t >> 32, 0, 0)), the word of
 *              orc_token_threshold: its 24-bit threshold truncated to 16 bits);
 *   ORC_INDEP: v = the upper 16 bits of element e = t N + n's word
 *              (word e mod 4 of Philox(counter = e / 4));
 *   ORC_RTNE:  round to nearest even (orc_float_to_bf16). */
int orc_sr_bf16_matrix(const float* X, int64_t T, int64_t N, int64_t ldx, int64_t t0, int mode, uint64_t seed,
                       uint32_t tensor_id, uint16_t* Y) {
    if (T < 0 || N < 0 || ldx < N || t0 < 0) return ORC_ERR_ARG;
    if (mode != ORC_S3R && mode != ORC_INDEP && mode != ORC_RTNE) return ORC_ERR_ARG;
    uint32_t key[2] = {(uint32_t)seed, tensor_id};
    for (int64_t i = 0; i < T; ++i) {
        int64_t t = t0 + i;
        uint32_t out[4];
        uint32_t ctr[4] = {(uint32_t)t, (uint32_t)((uint64_t)t >> 32), 0u, 0u};
        orc_philox4x32_10(ctr, key, out);
        uint32_t v_tok = out[0] >> 16;
        for (int64_t n = 0; n < N; ++n) {
            float x = X[i * ldx + n];
            if (mode == ORC_RTNE) {
                Y[i * N + n] = orc_float_to_bf16(x);
                continue;
            }
            uint32_t v = v_tok;
            if (mode == ORC_INDEP) {
                uint64_t e = (uint64_t)t * (uint64_t)N + (uint64_t)n, c = e >> 2;
                uint32_t ce[4] = {(uint32_t)c, (uint32_t)(c >> 32), 0u, 0u}, w[4];
                orc_philox4x32_10(ce, key, w);
                v = w[e & 3u] >> 16;
            }
            Y[i * N + n] = orc_sr_bf16(x, v);
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Stochastic rounding of fp32 to FP8 e4m3 (1 sign, 4 exponent bits with     */
/* bias 7, 3 mantissa bits; no infinity, largest finite 448, 0x7F NaN), the   */
/* FP8 form of the same hardware conversion ([S3R] §II).  y = x * inv_scale   */
/* in fp32 first (the caller's scale).  On the magnitude m = |y|: the e4m3    */
/* spacing is s = 2^(e-3) for m in [2^e, 2^(e+1)), e >= -6, and 2^-9 below    */
/* 2^-6; with k = floor(m / s) and p = m / s - k, the magnitude becomes       */
/* (k + 1) s iff floor(p 2^16) > v for the 16-bit threshold v (probability    */
/* floor(p 2^16) / 2^16, [SRB] "The probability formula" to 2^-16).  m >= 448 */
/* (infinities included) saturates to 448; NaN gives 0x7F.  RTNE rounds to    */
/* nearest even and saturates the same way.                                   */
/* ------------------------------------------------------------------------- */
static uint8_t orc_e4m3_round(float y, int mode, uint32_t v) {
    uint32_t u;
    memcpy(&u, &y, 4);
    uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
    uint32_t mag = u & 0x7FFFFFFFu;
    if (mag > 0x7F800000u) return 0x7Fu;
    double m = fabs((double)y);
    if (m >= 448.0) return (uint8_t)(sign | 0x7Eu);
    int e = 0;
    if (m > 0.0) {
        (void)frexp(m, &e);   /* m = f 2^e, f in [0.5, 1): the binade is 2^(e-1) */
        e -= 1;
    }
    int sub = (m < ldexp(1.0, -6));
    double s = sub ? ldexp(1.0, -9) : ldexp(1.0, e - 3);
    double q = m / s;                          /* exact: s is a power of two */
    int64_t k = (int64_t)floor(q);
    double p = q - (double)k;                  /* exact */
    if (mode == ORC_RTNE) {
        if (p > 0.5 || (p == 0.5 && (k & 1))) k += 1;
    } else {
        uint32_t f16 = (uint32_t)floor(p * 65536.0);
        if (f16 > (v & 0xFFFFu)) k += 1;
    }
    uint32_t bits;
    if (sub) {
        bits = (uint32_t)k;                    /* k <= 8: subnormal codes, 8 = 2^-6 */
    } else {
        bits = (uint32_t)(((e + 7) << 3) + (int)(k - 8));   /* k = 16 carries into the exponent */
    }
    if (bits > 0x7Eu) bits = 0x7Eu;            /* beyond 448: saturate */
    return (uint8_t)(sign | bits);
}

uint8_t orc_sr_e4m3(float y, uint32_t v) { return orc_e4m3_round(y, ORC_S3R, v); }
uint8_t orc_rn_e4m3(float y) { return orc_e4m3_round(y, ORC_RTNE, 0u); }

/* X [T, N] fp32 (row stride ldx) -> Y [T, N] e4m3 codes (row stride N):
 * y = x * inv_scale in fp32, then per mode as orc_sr_bf16_matrix (S3R: the
 * token word's upper 16 bits; INDEP: element e's word; RTNE). Row i is token t0 + i. */
int orc_sr_fp8_matrix(const float* X, int64_t T, int64_t N, int64_t ldx, int64_t t0, float inv_scale, int mode,
                      uint64_t seed, uint32_t tensor_id, uint8_t* Y) {
    if (T < 0 || N < 0 || ldx < N || t0 < 0) return ORC_ERR_ARG;
    if (mode != ORC_S3R && mode != ORC_INDEP && mode != ORC_RTNE) return ORC_ERR_ARG;
    uint32_t key[2] = {(uint32_t)seed, tensor_id};
    for (int64_t i = 0; i < T; ++i) {
        int64_t t = t0 + i;
        uint32_t out[4];
        uint32_t ctr[4] = {(uint32_t)t, (uint32_t)((uint64_t)t >> 32), 0u, 0u};
        orc_philox4x32_10(ctr, key, out);
        uint32_t v_tok = out[0] >> 16;
        for (int64_t n = 0; n < N; ++n) {
            float y = X[i * ldx + n] * inv_scale;
            uint32_t v = v_tok;
            if (mode == ORC_INDEP) {
                uint64_t e = (uint64_t)t * (uint64_t)N + (uint64_t)n, c = e >> 2;
                uint32_t ce[4] = {(uint32_t)c, (uint32_t)(c >> 32), 0u, 0u}, w[4];
                orc_philox4x32_10(ce, key, w);
                v = w[e & 3u] >> 16;
            }
            Y[i * N + n] = orc_e4m3_round(y, mode, v);
        }
    }
    return ORC_OK;
}
