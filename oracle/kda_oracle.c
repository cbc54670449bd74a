/*
 * kda_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * The plain, slow, fp64 CPU oracle for the Kimi Delta Attention (KDA) forward
 * pass. Only the tests, the package smoke check and the benchmark's CPU
 * baseline leg may load this code; the product path never does. It shares no
 * code, header, table or constant with the CUDA library.
 *
 * What it computes, per (sequence, head), token by token, with no chunking,
 * no base-2 rebasing and no approximation:
 *
 *   x_t[c]   = exp(A_log[h]) * (g_t[c] + dt_bias[h,c])   (A_log NULL -> factor 1,
 *                                                         dt_bias NULL -> bias 0)
 *   a_t[c]   = lower_bound * sigmoid(x_t[c])              natural-log gate
 *   alpha_t  = exp(a_t)            beta_t = sigmoid(beta logit_t)
 *   S_t      = S_{t-1} Diag(alpha_t) (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *   o_t      = scale * S_t q_t
 *
 * S is V x K, stored row-major [v][c] (K contiguous), like the state tensors.
 *
 * Sources (page title -- section):
 *  - gate: "FlashKDA lower_bound Parameter: Controlling Exponentiation
 *    Precision in Selective State Space Models" -- FAQ "How does lower_bound
 *    interact with dt_bias?" gives lower_bound * sigmoid(g_raw + dt_bias); the
 *    pages never say how A_log enters. Reading adopted: A_log multiplies the
 *    biased gate through exp(A_log[h]) (the common KDA/Mamba parameterisation).
 *    The base-2 rebasing of "Base-2 Exponent Optimization in FlashKDA" --
 *    "Re-basing the Gate Activation" is exact in real arithmetic, so the oracle
 *    keeps natural exponentials.
 *  - beta: "FlashKDA Input Tensor Shapes and DTypes" -- "Gating Tensors and
 *    Output Buffer" (a sigmoid is applied to the beta logits).
 *  - scale: same page, "Global Scaling Factor" (a plain multiplicative factor;
 *    it is linear, so it is applied to the output).
 *  - recurrence: the pages name Kimi Delta Attention but never print its state
 *    update; this is the gated delta rule with a per-channel (diagonal) decay,
 *    the published definition of KDA.
 *  - states and varlen: "FlashKDA Input Tensor Shapes and DTypes" -- "Initial
 *    and Final States" and "Variable-Length Mode". Each varlen sequence starts
 *    from its own initial state.
 *
 * bf16 inputs arrive as raw 16-bit patterns and are widened exactly.
 *
 * Optional (qk_l2norm != 0): every (token, head) vector of q and k is first
 * L2-normalised, x[c] <- x[c] / sqrt(sum_c' x[c']^2 + 1e-6). The pages do not
 * say whether q and k arrive normalised (their examples draw them from randn);
 * this option is the library's KDA_FLAG_QK_L2NORM, with the epsilon placed
 * inside the square root.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double widen_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double sigmoid(double x)
{
    return 1.0 / (1.0 + exp(-x));
}

/* One token of the recurrence on one V x K state (row-major [v][c]).
 * pred is scratch of length V. */
static void token_step(double *S, int K, int V, const double *alpha, double beta,
                       const double *k, const double *v, const double *q,
                       double scale, double *o, double *pred)
{
    /* S <- S Diag(alpha): column c is scaled by alpha[c]. */
    for (int r = 0; r < V; r++)
        for (int c = 0; c < K; c++)
            S[(size_t)r * K + c] *= alpha[c];
    /* pred = S k (the state's prediction of v for key k). */
    for (int r = 0; r < V; r++) {
        double s = 0.0;
        for (int c = 0; c < K; c++)
            s += S[(size_t)r * K + c] * k[c];
        pred[r] = s;
    }
    /* S (I - beta k k^T) + beta v k^T  =  S + beta (v - S k) k^T. */
    for (int r = 0; r < V; r++) {
        double e = beta * (v[r] - pred[r]);
        for (int c = 0; c < K; c++)
            S[(size_t)r * K + c] += e * k[c];
    }
    /* o = scale * S q, with S the state after this token. */
    for (int r = 0; r < V; r++) {
        double s = 0.0;
        for (int c = 0; c < K; c++)
            s += S[(size_t)r * K + c] * q[c];
        o[r] = scale * s;
    }
}

/* Number of independent (sequence, head) units and, for unit u, its token
 * range [t0, t1) in the flattened token axis and its state slot. */
static void unit_span(int u, int H, int T, const int64_t *cu, int *slot,
                      int64_t *t0, int64_t *t1)
{
    int seq = u / H;
    if (cu) {
        *t0 = cu[seq];
        *t1 = cu[seq + 1];
    } else {
        *t0 = (int64_t)seq * T;
        *t1 = (int64_t)seq * T + T;
    }
    *slot = seq;
}

static int check_common(int B, int T, int H, int K, int V, int N,
                        const int64_t *cu)
{
    if (B < 0 || T < 0 || H <= 0 || K <= 0 || V <= 0)
        return -1;
    if (cu) {
        if (B != 1 || N < 1)
            return -1;
        if (cu[0] != 0 || cu[N] != T)
            return -1;
        for (int i = 0; i < N; i++)
            if (cu[i + 1] < cu[i])
                return -1;
    }
    return 0;
}

/*
 * Gate only: a[t,h,c] = lower_bound * sigmoid(exp(A_log[h]) (g + dt_bias[h,c])),
 * natural-log units. g: [n_tok, H, K] bf16 bits; out: same shape, fp64.
 */
int kda_oracle_gate(const uint16_t *g, const float *A_log, const float *dt_bias,
                    double lower_bound, double *out, int64_t n_tok, int H, int K)
{
    if (!g || !out || H <= 0 || K <= 0 || n_tok < 0)
        return -1;
    for (int64_t t = 0; t < n_tok; t++)
        for (int h = 0; h < H; h++) {
            double a = A_log ? exp((double)A_log[h]) : 1.0;
            for (int c = 0; c < K; c++) {
                size_t i = ((size_t)t * H + h) * K + c;
                double b = dt_bias ? (double)dt_bias[(size_t)h * K + c] : 0.0;
                out[i] = lower_bound * sigmoid(a * (widen_bf16(g[i]) + b));
            }
        }
    return 0;
}

/*
 * Full forward from the library's inputs.
 *   q, k, g: [B, T, H, K] bf16 bits;  v: [B, T, H, V] bf16 bits;
 *   beta: [B, T, H] bf16 bits (logits);  A_log: [H] fp32 or NULL;
 *   dt_bias: [H, K] fp32 or NULL;  out: [B, T, H, V] fp64;
 *   initial_state / final_state: [B|N, H, V, K] fp64 or NULL;
 *   cu_seqlens: [N+1] or NULL (then B == 1 and T is the packed length).
 *   qk_l2norm: nonzero to L2-normalise q and k per (token, head) first.
 * Returns 0, or -1 on bad arguments.
 */
int kda_oracle_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                   const uint16_t *g, const uint16_t *beta, double scale,
                   double *out, const float *A_log, const float *dt_bias,
                   double lower_bound, const double *initial_state,
                   double *final_state, const int64_t *cu_seqlens, int B, int T,
                   int H, int K, int V, int N, int qk_l2norm, int nthreads)
{
    if (!q || !k || !v || !g || !beta || !out)
        return -1;
    if (check_common(B, T, H, K, V, N, cu_seqlens))
        return -1;
    int nseq = cu_seqlens ? N : B;
    int nunits = nseq * H;
    if (nthreads < 1)
        nthreads = 1;
    int bad = 0;

#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : bad)
    for (int u = 0; u < nunits; u++) {
        int h = u % H, slot;
        int64_t t0, t1;
        unit_span(u, H, T, cu_seqlens, &slot, &t0, &t1);
        double *S = calloc((size_t)V * K, sizeof(double));
        double *buf = malloc(sizeof(double) * (size_t)(4 * K + 2 * V));
        if (!S || !buf) {
            free(S);
            free(buf);
            bad |= 1;
            continue;
        }
        double *alpha = buf, *kk = buf + K, *qq = buf + 2 * K,
               *xg = buf + 3 * K, *vv = buf + 4 * K, *pred = buf + 4 * K + V;
        size_t sbase = ((size_t)slot * H + h) * (size_t)V * K;
        if (initial_state)
            memcpy(S, initial_state + sbase, sizeof(double) * (size_t)V * K);
        double a = A_log ? exp((double)A_log[h]) : 1.0;
        for (int64_t t = t0; t < t1; t++) {
            size_t rk = ((size_t)t * H + h) * K, rv = ((size_t)t * H + h) * V;
            for (int c = 0; c < K; c++) {
                double b = dt_bias ? (double)dt_bias[(size_t)h * K + c] : 0.0;
                xg[c] = a * (widen_bf16(g[rk + c]) + b);
                alpha[c] = exp(lower_bound * sigmoid(xg[c]));
                kk[c] = widen_bf16(k[rk + c]);
                qq[c] = widen_bf16(q[rk + c]);
            }
            if (qk_l2norm) {
                double sk = 0.0, sq = 0.0;
                for (int c = 0; c < K; c++) {
                    sk += kk[c] * kk[c];
                    sq += qq[c] * qq[c];
                }
                double fk = 1.0 / sqrt(sk + 1e-6), fq = 1.0 / sqrt(sq + 1e-6);
                for (int c = 0; c < K; c++) {
                    kk[c] *= fk;
                    qq[c] *= fq;
                }
            }
            for (int r = 0; r < V; r++)
                vv[r] = widen_bf16(v[rv + r]);
            double bt = sigmoid(widen_bf16(beta[(size_t)t * H + h]));
            token_step(S, K, V, alpha, bt, kk, vv, qq, scale, out + rv, pred);
        }
        if (final_state)
            memcpy(final_state + sbase, S, sizeof(double) * (size_t)V * K);
        free(S);
        free(buf);
    }
    return bad ? -1 : 0;
}

/*
 * The recurrence alone, from already-activated quantities, all fp64:
 *   q, k, alpha: [B, T, H, K];  v, out: [B, T, H, V];  beta: [B, T, H]
 *   (beta here is the activated value, not a logit).
 * Same state and varlen conventions as kda_oracle_fwd. Used by the exact
 * rational and closed-form checks, which need K and V other than 128.
 */
int kda_oracle_core(const double *q, const double *k, const double *v,
                    const double *alpha, const double *beta, double scale,
                    double *out, const double *initial_state, double *final_state,
                    const int64_t *cu_seqlens, int B, int T, int H, int K, int V,
                    int N, int nthreads)
{
    if (!q || !k || !v || !alpha || !beta || !out)
        return -1;
    if (check_common(B, T, H, K, V, N, cu_seqlens))
        return -1;
    int nseq = cu_seqlens ? N : B;
    int nunits = nseq * H;
    if (nthreads < 1)
        nthreads = 1;
    int bad = 0;

#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : bad)
    for (int u = 0; u < nunits; u++) {
        int h = u % H, slot;
        int64_t t0, t1;
        unit_span(u, H, T, cu_seqlens, &slot, &t0, &t1);
        double *S = calloc((size_t)V * K, sizeof(double));
        double *pred = malloc(sizeof(double) * (size_t)V);
        if (!S || !pred) {
            free(S);
            free(pred);
            bad |= 1;
            continue;
        }
        size_t sbase = ((size_t)slot * H + h) * (size_t)V * K;
        if (initial_state)
            memcpy(S, initial_state + sbase, sizeof(double) * (size_t)V * K);
        for (int64_t t = t0; t < t1; t++) {
            size_t rk = ((size_t)t * H + h) * K, rv = ((size_t)t * H + h) * V;
            token_step(S, K, V, alpha + rk, beta[(size_t)t * H + h], k + rk,
                       v + rv, q + rk, scale, out + rv, pred);
        }
        if (final_state)
            memcpy(final_state + sbase, S, sizeof(double) * (size_t)V * K);
        free(S);
        free(pred);
    }
    return bad ? -1 : 0;
}
