/*
 * KDA oracle: a plain, slow, obviously correct fp64 CPU implementation of the
 * Kimi Delta Attention gated delta-rule recurrence.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the bench's CPU
 * baseline may load this file's library. It shares no code, header or constant
 * with the CUDA path.
 *
 * What it computes, per token t of a sequence and per head h (the update the
 * vLLM pages call the "KDA recurrence": PR #60683 "specialized decode for
 * Kimi-K3", section Purpose; the packed decode call of PR #51682, section
 * "key source excerpts"):
 *   x_c   = raw_g[t,h,c] + dt_bias[h,c]
 *   g_c   = -exp(A_log[h]) * softplus(x_c)                  (no lower bound)
 *         =  lower_bound * sigmoid(exp(A_log[h]) * x_c)      (lower bound set)
 *   beta  = sigmoid(raw_beta[t,h])
 *   q^    = scale * q / sqrt(|q|^2 + eps),  k^ = k / sqrt(|k|^2 + eps)
 *   S    <- Diag(exp(g)) S
 *   u     = beta * (v - S^T k^)
 *   S    <- S + k^ u^T
 *   o     = S^T q^
 * which is S_t = (I - beta k^ k^T) Diag(alpha) S_{t-1} + beta k^ v^T, o_t = S_t^T q^.
 * The gate formula is a documented reading (the pages name raw_g, A_log,
 * dt_bias and lower_bound as the gate's inputs but print no formula).
 *
 * A second routine evaluates the same result in the chunked (WY) form that
 * chunk_kda_with_fused_gate / recompute_w_u use (PR #50649, section Purpose):
 * in-chunk cumulative log-decay b, the strictly lower A, T = (I + A)^-1,
 * W = T diag(beta) (K^ * e^b), U~ = T diag(beta) V, U = U~ - W S0,
 * O = (Q^ * e^b) S0 + Aqk U, S_C = Diag(e^{b_C}) S0 + (K^ * e^{b_C - b})^T U.
 * Every pairwise decay e^{b_r - b_i} is evaluated directly (no factoring), so it
 * cannot overflow. It exists to pin the chunk algorithm against the sequential
 * definition.
 *
 * Layouts (as the library's): mixed_qkv bf16 bits [N, ld_qkv] with row
 * [q(H*K) | k(H*K) | v(H*V)], raw_g bf16 [N, ld_g] (H*K used), raw_beta bf16
 * [N, ld_beta] (H used), A_log f32 [H], dt_bias f32 [H*K] or NULL, states
 * [K][V] row-major per (sequence, head).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_f64(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double softplus(double x)
{
    /* log(1 + e^x) without overflow */
    return fmax(x, 0.0) + log1p(exp(-fabs(x)));
}

static double sigmoid(double y)
{
    return 1.0 / (1.0 + exp(-y));
}

/* The per-channel log-decay g (<= 0) of one (token, head, channel). */
static double gate_log_decay(double raw_g, double dt_bias, double A_log,
                             int has_lower_bound, double lower_bound)
{
    double x = raw_g + dt_bias;
    if (has_lower_bound)
        return lower_bound * sigmoid(exp(A_log) * x);
    return -exp(A_log) * softplus(x);
}

typedef struct {
    int H, K, V;
    const float *A_log;
    const float *dt_bias;
    int has_lower_bound;
    double lower_bound, scale, eps;
    const double *qkv64;   /* if set: q/k/v rows are fp64 values here (pitch ld64), not bf16 */
    int64_t ld64;
} heads_t;

/* Element `i` of the q|k|v row of token t: bf16 bits, or fp64 when hp->qkv64 is set. */
static double qkv_at(const heads_t *hp, const uint16_t *mixed_qkv, int64_t ld_qkv, int64_t t,
                     size_t i)
{
    if (hp->qkv64)
        return hp->qkv64[t * hp->ld64 + (int64_t)i];
    return bf16_to_f64(mixed_qkv[t * ld_qkv + (int64_t)i]);
}

/* Reads one token's q^, k^ (normalised, q^ scaled), v, g, beta for head h. */
static void load_token(const heads_t *hp, const uint16_t *mixed_qkv, int64_t ld_qkv, int64_t t,
                       const uint16_t *g_row, const uint16_t *beta_row, int h, double *qh,
                       double *kh, double *v, double *g, double *beta)
{
    int K = hp->K, V = hp->V, H = hp->H;
    size_t q0 = (size_t)h * K, k0 = (size_t)H * K + (size_t)h * K;
    size_t v0 = 2 * (size_t)H * K + (size_t)h * V;
    double qn = 0.0, kn = 0.0;
    for (int c = 0; c < K; c++) {
        qh[c] = qkv_at(hp, mixed_qkv, ld_qkv, t, q0 + c);
        kh[c] = qkv_at(hp, mixed_qkv, ld_qkv, t, k0 + c);
        qn += qh[c] * qh[c];
        kn += kh[c] * kh[c];
    }
    double qs = hp->scale / sqrt(qn + hp->eps);
    double ks = 1.0 / sqrt(kn + hp->eps);
    for (int c = 0; c < K; c++) {
        qh[c] *= qs;
        kh[c] *= ks;
    }
    for (int j = 0; j < V; j++)
        v[j] = qkv_at(hp, mixed_qkv, ld_qkv, t, v0 + j);
    for (int c = 0; c < K; c++) {
        double db = hp->dt_bias ? (double)hp->dt_bias[(size_t)h * K + c] : 0.0;
        g[c] = gate_log_decay(bf16_to_f64(g_row[(size_t)h * K + c]), db,
                              (double)hp->A_log[h], hp->has_lower_bound, hp->lower_bound);
    }
    *beta = sigmoid(bf16_to_f64(beta_row[h]));
}

/* ---- gate ------------------------------------------------------------------ */

/* g_out [N, H*K] and beta_out [N, H], fp64. */
void kda_oracle_gate(const uint16_t *raw_g, int64_t ld_g, const uint16_t *raw_beta,
                     int64_t ld_beta, int64_t N, int H, int K, const float *A_log,
                     const float *dt_bias, int has_lower_bound, double lower_bound,
                     double *g_out, double *beta_out)
{
    for (int64_t t = 0; t < N; t++) {
        for (int h = 0; h < H; h++) {
            for (int c = 0; c < K; c++) {
                double db = dt_bias ? (double)dt_bias[(size_t)h * K + c] : 0.0;
                g_out[t * (int64_t)H * K + (int64_t)h * K + c] =
                    gate_log_decay(bf16_to_f64(raw_g[t * ld_g + (int64_t)h * K + c]), db,
                                   (double)A_log[h], has_lower_bound, lower_bound);
            }
            beta_out[t * H + h] = sigmoid(bf16_to_f64(raw_beta[t * ld_beta + h]));
        }
    }
}

/* ---- sequential recurrence --------------------------------------------------- */

/* One (sequence, head): tokens [t0, t1). S is [K][V] in/out (fp64). Writes o rows
 * out[t, h*V + j] (fp64, row pitch ld_out). */
static void recur_one(const heads_t *hp, const uint16_t *mixed_qkv, int64_t ld_qkv,
                      const uint16_t *raw_g, int64_t ld_g, const uint16_t *raw_beta,
                      int64_t ld_beta, int64_t t0, int64_t t1, int h, double *S,
                      double *out, int64_t ld_out, double *ckpt, int64_t ckpt_stride)
{
    int K = hp->K, V = hp->V;
    double *qh = malloc(sizeof(double) * K), *kh = malloc(sizeof(double) * K);
    double *g = malloc(sizeof(double) * K), *v = malloc(sizeof(double) * V);
    double *u = malloc(sizeof(double) * V);
    double beta;
    for (int64_t t = t0; t < t1; t++) {
        load_token(hp, mixed_qkv, ld_qkv, t, raw_g + t * ld_g, raw_beta + t * ld_beta, h,
                   qh, kh, v, g, &beta);
        /* S <- Diag(exp(g)) S */
        for (int c = 0; c < K; c++) {
            double a = exp(g[c]);
            for (int j = 0; j < V; j++)
                S[(size_t)c * V + j] *= a;
        }
        /* u = beta (v - S^T k^) */
        for (int j = 0; j < V; j++) {
            double acc = 0.0;
            for (int c = 0; c < K; c++)
                acc += S[(size_t)c * V + j] * kh[c];
            u[j] = beta * (v[j] - acc);
        }
        /* S <- S + k^ u^T */
        for (int c = 0; c < K; c++)
            for (int j = 0; j < V; j++)
                S[(size_t)c * V + j] += kh[c] * u[j];
        /* o = S^T q^ */
        for (int j = 0; j < V; j++) {
            double acc = 0.0;
            for (int c = 0; c < K; c++)
                acc += S[(size_t)c * V + j] * qh[c];
            out[t * ld_out + (int64_t)h * V + j] = acc;
        }
        /* optional copy of the state after this token */
        if (ckpt)
            memcpy(ckpt + (t - t0) * ckpt_stride, S, sizeof(double) * (size_t)K * V);
    }
    free(qh); free(kh); free(g); free(v); free(u);
}

/*
 * Runs the recurrence for `num_seqs` sequences whose rows are
 * [row_begin[s], row_end[s]). states: [num_seqs][H][K][V] fp64, in/out.
 * out: [N][ld_out] fp64 (only the processed rows and heads are written).
 * Heads outside [head_lo, head_hi) are skipped (used to sample large cases).
 * nthreads <= 0 uses the OpenMP default.
 */
void kda_oracle_recurrent(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                          int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
                          const int64_t *row_begin, const int64_t *row_end, int64_t num_seqs,
                          int H, int K, int V, const float *A_log, const float *dt_bias,
                          int has_lower_bound, double lower_bound, double scale, double eps,
                          double *states, double *out, int64_t ld_out, int head_lo,
                          int head_hi, int nthreads)
{
    heads_t hp = {H, K, V, A_log, dt_bias, has_lower_bound, lower_bound, scale, eps, NULL, 0};
    int64_t nh = head_hi - head_lo;
    int64_t work = num_seqs * nh;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t w = 0; w < work; w++) {
        int64_t s = w / nh;
        int h = head_lo + (int)(w % nh);
        double *S = states + ((size_t)s * H + h) * (size_t)K * V;
        recur_one(&hp, mixed_qkv, ld_qkv, raw_g, ld_g, raw_beta, ld_beta, row_begin[s],
                  row_end[s], h, S, out, ld_out, NULL, 0);
    }
}

/*
 * As kda_oracle_recurrent over all heads, and also records the state after every token:
 * ckpt is [num_seqs][Tmax][H][K][V] fp64; the state of sequence s, head h after its
 * t-th token (t < row_end - row_begin <= Tmax) is ckpt[((s*Tmax + t)*H + h)*K*V ...].
 */
void kda_oracle_recurrent_ckpt(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                               int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
                               const int64_t *row_begin, const int64_t *row_end, int64_t num_seqs,
                               int H, int K, int V, const float *A_log, const float *dt_bias,
                               int has_lower_bound, double lower_bound, double scale, double eps,
                               double *states, double *out, int64_t ld_out, double *ckpt,
                               int64_t Tmax, int nthreads)
{
    heads_t hp = {H, K, V, A_log, dt_bias, has_lower_bound, lower_bound, scale, eps, NULL, 0};
    int64_t work = num_seqs * H;
    size_t KV = (size_t)K * V;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t w = 0; w < work; w++) {
        int64_t s = w / H;
        int h = (int)(w % H);
        double *S = states + ((size_t)s * H + h) * KV;
        recur_one(&hp, mixed_qkv, ld_qkv, raw_g, ld_g, raw_beta, ld_beta, row_begin[s],
                  row_end[s], h, S, out, ld_out, ckpt + ((size_t)s * Tmax * H + h) * KV,
                  (int64_t)H * (int64_t)KV);
    }
}

/*
 * kda_oracle_recurrent with fp64 q|k|v rows (qkv64 [N][ld64]) instead of bf16 bits: the
 * inputs of the recurrence when the short causal convolution runs in front of it.
 */
void kda_oracle_recurrent_f64in(const double *qkv64, int64_t ld64, const uint16_t *raw_g,
                                int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
                                const int64_t *row_begin, const int64_t *row_end,
                                int64_t num_seqs, int H, int K, int V, const float *A_log,
                                const float *dt_bias, int has_lower_bound, double lower_bound,
                                double scale, double eps, double *states, double *out,
                                int64_t ld_out, int nthreads)
{
    heads_t hp = {H, K, V, A_log, dt_bias, has_lower_bound, lower_bound, scale, eps, qkv64, ld64};
    int64_t work = num_seqs * H;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t w = 0; w < work; w++) {
        int64_t s = w / H;
        int h = (int)(w % H);
        double *S = states + ((size_t)s * H + h) * (size_t)K * V;
        recur_one(&hp, NULL, 0, raw_g, ld_g, raw_beta, ld_beta, row_begin[s], row_end[s], h, S,
                  out, ld_out, NULL, 0);
    }
}

int kda_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- chunked (WY) form ------------------------------------------------------------ */

static void chunk_one(const heads_t *hp, const uint16_t *mixed_qkv, int64_t ld_qkv,
                      const uint16_t *raw_g, int64_t ld_g, const uint16_t *raw_beta,
                      int64_t ld_beta, int64_t t0, int64_t t1, int h, int C, double *S,
                      double *out, int64_t ld_out)
{
    int K = hp->K, V = hp->V;
    size_t CK = (size_t)C * K, CV = (size_t)C * V;
    double *Q = malloc(sizeof(double) * CK), *Kh = malloc(sizeof(double) * CK);
    double *G = malloc(sizeof(double) * CK), *B = malloc(sizeof(double) * CK);
    double *Vv = malloc(sizeof(double) * CV), *beta = malloc(sizeof(double) * C);
    double *A = malloc(sizeof(double) * C * C), *Aqk = malloc(sizeof(double) * C * C);
    double *T = malloc(sizeof(double) * C * C);
    double *W = malloc(sizeof(double) * CK), *Ut = malloc(sizeof(double) * CV);
    double *U = malloc(sizeof(double) * CV), *O = malloc(sizeof(double) * CV);
    double *Snew = malloc(sizeof(double) * (size_t)K * V);

    for (int64_t c0 = t0; c0 < t1; c0 += C) {
        int n = (int)((t1 - c0) < C ? (t1 - c0) : C);
        for (int r = 0; r < n; r++)
            load_token(hp, mixed_qkv, ld_qkv, c0 + r, raw_g + (c0 + r) * ld_g,
                       raw_beta + (c0 + r) * ld_beta, h, Q + (size_t)r * K, Kh + (size_t)r * K,
                       Vv + (size_t)r * V, G + (size_t)r * K, &beta[r]);
        /* b_r = sum_{i<=r} g_i (in-chunk cumulative log-decay) */
        for (int c = 0; c < K; c++) {
            double acc = 0.0;
            for (int r = 0; r < n; r++) {
                acc += G[(size_t)r * K + c];
                B[(size_t)r * K + c] = acc;
            }
        }
        /* A[r,i] = beta_r sum_c k^_r k^_i e^{b_r - b_i}  (i < r);  Aqk for i <= r */
        for (int r = 0; r < n; r++) {
            for (int i = 0; i < n; i++) {
                double a = 0.0, aq = 0.0;
                if (i <= r) {
                    for (int c = 0; c < K; c++) {
                        double d = exp(B[(size_t)r * K + c] - B[(size_t)i * K + c]);
                        a += Kh[(size_t)r * K + c] * Kh[(size_t)i * K + c] * d;
                        aq += Q[(size_t)r * K + c] * Kh[(size_t)i * K + c] * d;
                    }
                }
                A[r * C + i] = (i < r) ? beta[r] * a : 0.0;
                Aqk[r * C + i] = (i <= r) ? aq : 0.0;
            }
        }
        /* T = (I + A)^-1 by forward substitution, column by column */
        for (int i = 0; i < n; i++) {
            for (int r = 0; r < n; r++) {
                double acc = (r == i) ? 1.0 : 0.0;
                for (int m = 0; m < r; m++)
                    acc -= A[r * C + m] * T[m * C + i];
                T[r * C + i] = acc;
            }
        }
        /* W = T diag(beta) (K^ * e^b),  U~ = T diag(beta) V */
        for (int r = 0; r < n; r++) {
            for (int c = 0; c < K; c++) {
                double acc = 0.0;
                for (int i = 0; i <= r; i++)
                    acc += T[r * C + i] * beta[i] * Kh[(size_t)i * K + c] * exp(B[(size_t)i * K + c]);
                W[(size_t)r * K + c] = acc;
            }
            for (int j = 0; j < V; j++) {
                double acc = 0.0;
                for (int i = 0; i <= r; i++)
                    acc += T[r * C + i] * beta[i] * Vv[(size_t)i * V + j];
                Ut[(size_t)r * V + j] = acc;
            }
        }
        /* U = U~ - W S0 */
        for (int r = 0; r < n; r++)
            for (int j = 0; j < V; j++) {
                double acc = 0.0;
                for (int c = 0; c < K; c++)
                    acc += W[(size_t)r * K + c] * S[(size_t)c * V + j];
                U[(size_t)r * V + j] = Ut[(size_t)r * V + j] - acc;
            }
        /* O = (Q^ * e^b) S0 + Aqk U */
        for (int r = 0; r < n; r++)
            for (int j = 0; j < V; j++) {
                double acc = 0.0;
                for (int c = 0; c < K; c++)
                    acc += Q[(size_t)r * K + c] * exp(B[(size_t)r * K + c]) * S[(size_t)c * V + j];
                for (int i = 0; i <= r; i++)
                    acc += Aqk[r * C + i] * U[(size_t)i * V + j];
                O[(size_t)r * V + j] = acc;
            }
        /* S_C = Diag(e^{b_last}) S0 + (K^ * e^{b_last - b})^T U */
        const double *bl = B + (size_t)(n - 1) * K;
        for (int c = 0; c < K; c++)
            for (int j = 0; j < V; j++) {
                double acc = exp(bl[c]) * S[(size_t)c * V + j];
                for (int i = 0; i < n; i++)
                    acc += Kh[(size_t)i * K + c] * exp(bl[c] - B[(size_t)i * K + c]) * U[(size_t)i * V + j];
                Snew[(size_t)c * V + j] = acc;
            }
        memcpy(S, Snew, sizeof(double) * (size_t)K * V);
        for (int r = 0; r < n; r++)
            for (int j = 0; j < V; j++)
                out[(c0 + r) * ld_out + (int64_t)h * V + j] = O[(size_t)r * V + j];
    }
    free(Q); free(Kh); free(G); free(B); free(Vv); free(beta); free(A); free(Aqk); free(T);
    free(W); free(Ut); free(U); free(O); free(Snew);
}

/* Same contract as kda_oracle_recurrent, evaluated chunk by chunk (chunk size C). */
void kda_oracle_chunked(const uint16_t *mixed_qkv, int64_t ld_qkv, const uint16_t *raw_g,
                        int64_t ld_g, const uint16_t *raw_beta, int64_t ld_beta,
                        const int64_t *row_begin, const int64_t *row_end, int64_t num_seqs,
                        int H, int K, int V, const float *A_log, const float *dt_bias,
                        int has_lower_bound, double lower_bound, double scale, double eps,
                        int C, double *states, double *out, int64_t ld_out, int nthreads)
{
    heads_t hp = {H, K, V, A_log, dt_bias, has_lower_bound, lower_bound, scale, eps, NULL, 0};
    int64_t work = num_seqs * H;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t w = 0; w < work; w++) {
        int64_t s = w / H;
        int h = (int)(w % H);
        double *S = states + ((size_t)s * H + h) * (size_t)K * V;
        chunk_one(&hp, mixed_qkv, ld_qkv, raw_g, ld_g, raw_beta, ld_beta, row_begin[s],
                  row_end[s], h, C, S, out, ld_out);
    }
}
