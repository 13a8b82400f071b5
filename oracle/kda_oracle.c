/*
 * fp64 CPU oracle for the KDA bounded-gate recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg load this library.  It shares no code, header, table or
 * helper with the CUDA path.
 *
 * What is computed, per sequence n, head h, and token t in token order (all
 * arithmetic in double precision; bf16 inputs are widened exactly):
 *
 *   q^ = q / sqrt(sum_c q_c^2 + eps),  k^ likewise
 *       -- "in-kernel q/k l2norm" (vLLM PR #55737 "Use FlashKDA for KDA
 *          chunked prefill", PR summary and Purpose).  eps is not printed on
 *          the pages; the caller passes it (1e-6 is the adopted reading).
 *   beta = 1 / (1 + exp(-beta_logit))
 *       -- "raw beta logits" enter the kernel and the sigmoid is applied
 *          inside it (same PR, summary: "pre-sigmoid beta cast no longer
 *          needed").
 *   lambda_c = lower_bound * sigmoid(exp(A_log[h]) * (g_c + dt_bias[h][c]))
 *       -- the bounded gate, printed verbatim in the same PR summary.  It is
 *          a per-channel log-decay: alpha_c = exp(lambda_c), lower_bound < 0.
 *   S <- Diag(alpha) S                      (decay of the dk rows of S)
 *   u  = beta * (v - S^T k^)                (delta-rule correction)
 *   S <- S + k^ u^T
 *   o  = scale * S^T q^
 *
 * The three state lines are the KDA delta rule
 *   S_t = (I - beta k^ k^T) Diag(alpha) S_{t-1} + beta k^ v^T
 * that the pages call "the same bounded-gate KDA recurrence" (same PR,
 * summary); expanding the product gives exactly the decay / correction /
 * rank-1 update above.  The output is read from the updated state S_t.
 *
 * State layout: S is dk x dv, row-major (dv fastest), o = S^T q^ has dv
 * entries.  Verify semantics ("seeds ... with the pool state and writes step
 * t's state to row (b, t)", TensorRT-LLM PR #21179 "GLM-5.3-Flash FP8
 * performance fixes on Hopper", KDA verify commit): the per-step state
 * record for token t is the state after token t.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* element-level definitions                                                  */
/* ------------------------------------------------------------------------- */

static double bf16_to_double(uint16_t h)
{
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* x^ = x / sqrt(sum x^2 + eps) over the d channels of one (token, head). */
void kda_oracle_l2norm(const double *x, int d, double eps, double *out)
{
    double ss = 0.0;
    for (int c = 0; c < d; ++c) ss += x[c] * x[c];
    double inv = 1.0 / sqrt(ss + eps);
    for (int c = 0; c < d; ++c) out[c] = x[c] * inv;
}

/*
 * Sigmoid-gated RMSNorm of output rows ("sigmoid RMSNorm" / "gated norm" on
 * BF16, D = 128 rows: sglang PR #42489 "Improve GLM-5.3-Flash DFlash decoding
 * on B300", Modifications and review thread; its kernel checks compare the
 * output and rstd).  The pages print no formula; the reading taken: per row
 * of d channels (one token and head), the row is normalised first and gated
 * after,
 *   rstd = 1 / sqrt(mean_c x_c^2 + eps)
 *   y_c  = x_c * rstd * w_c * sigmoid(z_c)
 * with the weight w shared by the heads and z the bf16 gate row.
 */
void kda_oracle_gated_rmsnorm(const double *x, const uint16_t *z, const double *w, double eps,
                              int rows, int d, double *y, double *rstd)
{
    for (int r = 0; r < rows; ++r) {
        const double *xr = x + (size_t)r * d;
        double ms = 0.0;
        for (int c = 0; c < d; ++c) ms += xr[c] * xr[c];
        ms /= d;
        double inv_rms = 1.0 / sqrt(ms + eps);
        rstd[r] = inv_rms;
        for (int c = 0; c < d; ++c)
            y[(size_t)r * d + c] = xr[c] * inv_rms * w[c] * sigmoid(bf16_to_double(z[(size_t)r * d + c]));
    }
}

/*
 * Short causal depthwise convolution of one input row ("three short
 * convolutions" on q, k and v per step, with per-step windows:
 * TensorRT-LLM PR #21179 "GLM-5.3-Flash FP8 performance fixes on Hopper",
 * KDA verify commit).  The pages print neither the width nor an activation;
 * the reading taken: W taps per channel, tap W-1 on the current input and tap
 * j on the input W-1-j tokens back,
 *   y_c = act( sum_{j<W-1} w_c[j] win[j]_c + w_c[W-1] x_c ),  act = SiLU or none,
 * where win holds the W-1 previous inputs of the sequence, oldest first
 * (seeded from the carried window, zero for a fresh sequence).  The window
 * then drops its oldest row and appends x.
 */
void kda_oracle_conv_step(double *win, const double *x, const double *w, int W, int d, int silu, double *y)
{
    for (int c = 0; c < d; ++c) {
        double acc = w[(size_t)c * W + (W - 1)] * x[c];
        for (int j = 0; j < W - 1; ++j) acc += w[(size_t)c * W + j] * win[(size_t)j * d + c];
        y[c] = silu ? acc * sigmoid(acc) : acc;
    }
    for (int j = 0; j + 1 < W - 1; ++j)
        for (int c = 0; c < d; ++c) win[(size_t)j * d + c] = win[(size_t)(j + 1) * d + c];
    if (W > 1)
        for (int c = 0; c < d; ++c) win[(size_t)(W - 2) * d + c] = x[c];
}

/* lambda_c = lower_bound * sigmoid(exp(A_log) * (g_c + dt_bias_c)). */
void kda_oracle_gate(const double *g, const double *dt_bias, double A_log,
                     double lower_bound, int d, double *lambda)
{
    double a = exp(A_log);
    for (int c = 0; c < d; ++c) lambda[c] = lower_bound * sigmoid(a * (g[c] + dt_bias[c]));
}

/*
 * One token of the recurrence on a dk x dv state.
 *   lambda: per-channel log-decay (dk), beta: scalar in [0, 1].
 *   qh, kh: already normalised query/key (dk), v: value (dv).
 *   o: output (dv).  S is updated in place.
 */
void kda_oracle_step(double *S, int dk, int dv, const double *qh, const double *kh,
                     const double *v, const double *lambda, double beta,
                     double scale, double *o)
{
    /* S <- Diag(alpha) S */
    for (int c = 0; c < dk; ++c) {
        double alpha = exp(lambda[c]);
        double *row = S + (size_t)c * dv;
        for (int j = 0; j < dv; ++j) row[j] *= alpha;
    }
    /* u = beta (v - S^T k^) */
    double u[dv];
    for (int j = 0; j < dv; ++j) {
        double w = 0.0;
        for (int c = 0; c < dk; ++c) w += S[(size_t)c * dv + j] * kh[c];
        u[j] = beta * (v[j] - w);
    }
    /* S <- S + k^ u^T */
    for (int c = 0; c < dk; ++c) {
        double *row = S + (size_t)c * dv;
        for (int j = 0; j < dv; ++j) row[j] += kh[c] * u[j];
    }
    /* o = scale S^T q^ */
    for (int j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int c = 0; c < dk; ++c) acc += S[(size_t)c * dv + j] * qh[c];
        o[j] = scale * acc;
    }
}

/*
 * Core recurrence for one (sequence, head) with the decay and beta given
 * directly (no gate, no normalisation): used to pin the recurrence on cases
 * the gate cannot produce exactly (alpha = 1, beta = 1).
 *   qh, kh: [T, dk]; v: [T, dv]; lambda: [T, dk]; beta: [T]
 *   S: [dk, dv] in/out; out: [T, dv]; step_states: [T, dk, dv] or NULL.
 */
int kda_oracle_core(const double *qh, const double *kh, const double *v,
                    const double *lambda, const double *beta, int T, int dk, int dv,
                    double scale, double *S, double *out, double *step_states)
{
    if (T < 0 || dk <= 0 || dv <= 0) return 1;
    for (int t = 0; t < T; ++t) {
        kda_oracle_step(S, dk, dv, qh + (size_t)t * dk, kh + (size_t)t * dk,
                        v + (size_t)t * dv, lambda + (size_t)t * dk, beta[t], scale,
                        out + (size_t)t * dv);
        if (step_states)
            memcpy(step_states + (size_t)t * dk * dv, S, sizeof(double) * (size_t)dk * dv);
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* full path over packed varlen sequences and heads                          */
/* ------------------------------------------------------------------------- */

typedef struct {
    const uint16_t *q, *k, *v, *g, *beta;
    const float *A_log, *dt_bias;
    double lower_bound, scale, eps;
    const int32_t *cu_seqlens;
    int num_seqs, H, dk, dv, head_begin, head_end;
    const double *S0;
    double *out, *S_final, *step_states;
    /* optional short convolution of q, k, v (dk == dv == d): weights [3][H][d][W]; windows [.][3][W-1][H][d] */
    const double *conv_w;
    int conv_W, conv_silu;
    const double *conv_win0;   /* [num_seqs] initial windows, or NULL (zero) */
    double *conv_win_final;    /* [num_seqs] final windows, or NULL */
    double *conv_win_steps;    /* [T_total] window after each token, or NULL */
    int next_task; /* shared task counter */
} job_t;

static void run_task(const job_t *J, int n, int h)
{
    const int dk = J->dk, dv = J->dv, H = J->H;
    const size_t state_elems = (size_t)dk * dv;
    double *S = (double *)calloc(state_elems, sizeof(double));
    double *x = (double *)malloc(sizeof(double) * (size_t)(dk > dv ? dk : dv));
    double *qh = (double *)malloc(sizeof(double) * (size_t)dk);
    double *kh = (double *)malloc(sizeof(double) * (size_t)dk);
    double *vv = (double *)malloc(sizeof(double) * (size_t)dv);
    double *gg = (double *)malloc(sizeof(double) * (size_t)dk);
    double *dtb = (double *)malloc(sizeof(double) * (size_t)dk);
    double *lam = (double *)malloc(sizeof(double) * (size_t)dk);

    if (J->S0) memcpy(S, J->S0 + ((size_t)n * H + h) * state_elems, sizeof(double) * state_elems);
    for (int c = 0; c < dk; ++c) dtb[c] = (double)J->dt_bias[(size_t)h * dk + c];
    const double A_log = (double)J->A_log[h];

    /* short convolution windows of this (sequence, head): [3][W-1][d] */
    const int W = J->conv_w ? J->conv_W : 0, d = dk;
    const size_t win_rows = W > 1 ? (size_t)(W - 1) : 0;
    double *win = W ? (double *)calloc(3 * win_rows * (size_t)d + 1, sizeof(double)) : NULL;
    double *raw = W ? (double *)malloc(sizeof(double) * (size_t)d) : NULL;
    if (W && J->conv_win0)
        for (int m = 0; m < 3; ++m)
            for (size_t j = 0; j < win_rows; ++j)
                memcpy(win + ((size_t)m * win_rows + j) * d,
                       J->conv_win0 + ((((size_t)n * 3 + m) * win_rows + j) * H + h) * d, sizeof(double) * d);

    for (int t = J->cu_seqlens[n]; t < J->cu_seqlens[n + 1]; ++t) {
        const size_t rk = ((size_t)t * H + h) * dk; /* row of q / k / g */
        const size_t rv = ((size_t)t * H + h) * dv; /* row of v / out   */
        if (W) {   /* q, k, v through their short convolutions, then as below */
            const uint16_t *src[3] = {J->q + rk, J->k + rk, J->v + rv};
            double *dst[3] = {x, kh, vv};
            for (int m = 0; m < 3; ++m) {
                for (int c = 0; c < d; ++c) raw[c] = bf16_to_double(src[m][c]);
                kda_oracle_conv_step(win + (size_t)m * win_rows * d, raw,
                                     J->conv_w + ((size_t)m * H + h) * d * W, W, d, J->conv_silu, dst[m]);
            }
            kda_oracle_l2norm(x, dk, J->eps, qh);
            memcpy(x, kh, sizeof(double) * dk);
            kda_oracle_l2norm(x, dk, J->eps, kh);
            if (J->conv_win_steps)
                for (int m = 0; m < 3; ++m)
                    for (size_t j = 0; j < win_rows; ++j)
                        memcpy(J->conv_win_steps + ((((size_t)t * 3 + m) * win_rows + j) * H + h) * d,
                               win + ((size_t)m * win_rows + j) * d, sizeof(double) * d);
        } else {
            for (int c = 0; c < dk; ++c) x[c] = bf16_to_double(J->q[rk + c]);
            kda_oracle_l2norm(x, dk, J->eps, qh);
            for (int c = 0; c < dk; ++c) x[c] = bf16_to_double(J->k[rk + c]);
            kda_oracle_l2norm(x, dk, J->eps, kh);
            for (int j = 0; j < dv; ++j) vv[j] = bf16_to_double(J->v[rv + j]);
        }
        for (int c = 0; c < dk; ++c) gg[c] = bf16_to_double(J->g[rk + c]);
        kda_oracle_gate(gg, dtb, A_log, J->lower_bound, dk, lam);
        double beta = sigmoid(bf16_to_double(J->beta[(size_t)t * H + h]));
        kda_oracle_step(S, dk, dv, qh, kh, vv, lam, beta, J->scale, J->out + rv);
        if (J->step_states)
            memcpy(J->step_states + ((size_t)t * H + h) * state_elems, S,
                   sizeof(double) * state_elems);
    }
    if (J->S_final)
        memcpy(J->S_final + ((size_t)n * H + h) * state_elems, S, sizeof(double) * state_elems);
    if (W && J->conv_win_final)
        for (int m = 0; m < 3; ++m)
            for (size_t j = 0; j < win_rows; ++j)
                memcpy(J->conv_win_final + ((((size_t)n * 3 + m) * win_rows + j) * H + h) * d,
                       win + ((size_t)m * win_rows + j) * d, sizeof(double) * d);
    free(S); free(x); free(qh); free(kh); free(vv); free(gg); free(dtb); free(lam); free(win); free(raw);
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    const int heads = J->head_end - J->head_begin;
    const int ntasks = J->num_seqs * heads;
    for (;;) {
        int i = __atomic_fetch_add(&J->next_task, 1, __ATOMIC_RELAXED);
        if (i >= ntasks) break;
        run_task(J, i / heads, J->head_begin + i % heads);
    }
    return NULL;
}

/*
 * Run every sequence of a packed varlen batch for heads [head_begin, head_end).
 *   q, k, g: bf16 bits [T_total, H, dk]; v: [T_total, H, dv]; beta_logits: [T_total, H]
 *   A_log: [H]; dt_bias: [H, dk]; cu_seqlens: [num_seqs + 1], non-decreasing, from 0
 *   S0: [num_seqs, H, dk, dv] or NULL (zero initial state)
 *   out: [T_total, H, dv]; S_final: [num_seqs, H, dk, dv] or NULL
 *   step_states: [T_total, H, dk, dv] or NULL (state after each token)
 * Only the selected heads' entries of out / S_final / step_states are written.
 * Returns 0, or 1 on invalid sizes.
 */
int kda_oracle_run_conv(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                        const uint16_t *g, const uint16_t *beta_logits,
                        const float *A_log, const float *dt_bias,
                        double lower_bound, double scale, double eps,
                        const int32_t *cu_seqlens, int num_seqs, int H, int dk, int dv,
                        int head_begin, int head_end, const double *S0,
                        double *out, double *S_final, double *step_states, int nthreads,
                        const double *conv_w, int conv_W, int conv_silu, const double *conv_win0,
                        double *conv_win_final, double *conv_win_steps);

int kda_oracle_run(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                   const uint16_t *g, const uint16_t *beta_logits,
                   const float *A_log, const float *dt_bias,
                   double lower_bound, double scale, double eps,
                   const int32_t *cu_seqlens, int num_seqs, int H, int dk, int dv,
                   int head_begin, int head_end, const double *S0,
                   double *out, double *S_final, double *step_states, int nthreads)
{
    return kda_oracle_run_conv(q, k, v, g, beta_logits, A_log, dt_bias, lower_bound, scale, eps, cu_seqlens,
                               num_seqs, H, dk, dv, head_begin, head_end, S0, out, S_final, step_states, nthreads,
                               NULL, 0, 0, NULL, NULL, NULL);
}

/*
 * kda_oracle_run with q, k and v first passed through their short causal
 * convolutions (kda_oracle_conv_step), when conv_w is not NULL:
 *   conv_w: [3 (q, k, v)][H][d][W]; conv_win0 / conv_win_final: [num_seqs][3][W-1][H][d]
 *   (initial windows or NULL for zero, final windows or NULL); conv_win_steps:
 *   [T_total][3][W-1][H][d] the window after each token, or NULL.  Needs dk == dv.
 */
int kda_oracle_run_conv(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                        const uint16_t *g, const uint16_t *beta_logits,
                        const float *A_log, const float *dt_bias,
                        double lower_bound, double scale, double eps,
                        const int32_t *cu_seqlens, int num_seqs, int H, int dk, int dv,
                        int head_begin, int head_end, const double *S0,
                        double *out, double *S_final, double *step_states, int nthreads,
                        const double *conv_w, int conv_W, int conv_silu, const double *conv_win0,
                        double *conv_win_final, double *conv_win_steps)
{
    if (num_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0) return 1;
    if (conv_w && (conv_W < 1 || dk != dv)) return 1;
    if (head_begin < 0 || head_end > H || head_begin > head_end) return 1;
    if (cu_seqlens[0] != 0) return 1;
    for (int n = 0; n < num_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return 1;
    job_t J = {q, k, v, g, beta_logits, A_log, dt_bias, lower_bound, scale, eps,
               cu_seqlens, num_seqs, H, dk, dv, head_begin, head_end, S0,
               out, S_final, step_states, conv_w, conv_W, conv_silu, conv_win0,
               conv_win_final, conv_win_steps, 0};
    if (nthreads < 1) nthreads = 1;
    if (nthreads == 1) {
        worker(&J);
        return 0;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int started = 0;
    for (int i = 0; i < nthreads; ++i)
        if (pthread_create(&th[started], NULL, worker, &J) == 0) ++started;
    if (started == 0) worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    return 0;
}
