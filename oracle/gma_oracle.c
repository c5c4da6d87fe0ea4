/*
 * fp64 CPU oracle for Gaussian Mixture Attention (GMA).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  The CUDA library
 * shares no code, header, table or helper with it.
 *
 * It states the method in its plain form, in double precision, one token at
 * a time, with no blocking, chunking or reordering.  Source: the GMA explainer
 * page "Gaussian Mixture Attention: Linear-Time Sequence Mixing via
 * Probabilistic Latent Routing", technical summary, sections
 * "핵심 메커니즘" (core mechanism) and "변형 및 학습" (variants and training):
 *
 *   S0  sigma^2 = softplus(raw variance), pi = softmax(mixture logits)
 *       ("변형 및 학습": reparameterisation, softplus for variances, softmax
 *       for priors).
 *   S1  gamma_{i,k} = p(z = k | x_i), the standard posterior of a GMM with
 *       means mu_k, diagonal covariances Sigma_k and priors pi_k
 *       ("핵심 메커니즘", probabilistic latent routing).  Q_X and K_X are routed
 *       through the same K components (the shared latent space).
 *   S2  write:  Vt = Gamma_K^T V,  Z = Gamma_K^T 1_N   ("핵심 메커니즘", write phase)
 *   S3  read:   O  = (Gamma_Q Vt) / (Gamma_Q Z + eps)  ("핵심 메커니즘", read phase)
 *   S4  causal: Vt and Z are prefix sums, O_i uses only j <= i
 *       ("변형 및 학습", bidirectional and causal variants)
 *   S5  decode: the causal recurrence advanced by one token (state updated
 *       with the token, then read).
 *   X   cross-attention ("의의 및 주장": cross-attention as an extension): the
 *       bidirectional write over N_k key/value rows, read by N_q query rows of
 *       another sequence.
 *   G   gradients ("변형 및 학습": the parameters are trained end to end by
 *       backpropagation, with softplus and softmax reparameterisations; "주요
 *       기여", gradient structure: the gradients pass through the
 *       responsibilities): dL/dO given, the gradients of Q_X, K_X, V, mu,
 *       the raw variances and the mixture logits, by the chain rule through
 *       the read, the write, the posterior and the reparameterisation.
 *   D   responsibility diagnostics ("결과 및 성능", interpretability: the
 *       components used, usage entropy, hard assignments): per head, the soft
 *       usage u_k = sum_i gamma_ik, the hard assignment argmax_k gamma_ik of
 *       every row (lowest k on ties) and its counts, and the entropies of the
 *       soft and hard usage distributions divided by log K.
 *
 * Readings where the page is silent (each is listed in the design notes):
 *   - one GMM per head, shared by Q_X and K_X and by every batch element;
 *   - the full Gaussian log-density, including the log(2 pi sigma^2) terms
 *     (the 2 pi term cancels in the posterior; it is kept here because this
 *     is the definition written out);
 *   - eps is added once to each row's scalar denominator Gamma_Q Z;
 *   - the causal prefix is inclusive (j <= i); a decode step writes the new
 *     token into the state before reading.
 *
 * Parity pins (tests that do not use this code): a library GMM posterior
 * (scikit-learn), the two-component logistic closed form, equal-component and
 * permutation identities, brute-force N x N affinity, rank(Gamma_Q Gamma_K^T)
 * <= K, causality under perturbation, K = 1 means, and sequence splitting.
 *
 * Layouts (row-major, double): per slice s the routing rows are x[s][n][d],
 * values v[s][n][dv], outputs out[s][n][dv]; a slice uses the parameters of
 * head head[s]: mu[h][k][d], var_raw[h][k][d], logit_pi[h][k].  A recurrent
 * state is state[s][K*dv + K]: the latent memory Vt[k][c] followed by Z[k].
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static const double kLog2Pi = 1.8378770664093454835606594728112; /* log(2 pi) */

int gma_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void gma_oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* softplus(r) = log(1 + e^r), evaluated without overflow. */
static double softplus(double r)
{
    return fmax(r, 0.0) + log1p(exp(-fabs(r)));
}

/* S0: variances of every head and log mixture priors (log-softmax of logits). */
void gma_oracle_params(int H, int K, int d, const double *var_raw, const double *logit_pi,
                       double *var, double *log_pi)
{
    for (long i = 0; i < (long)H * K * d; ++i)
        var[i] = softplus(var_raw[i]);
    for (int h = 0; h < H; ++h) {
        const double *l = logit_pi + (long)h * K;
        double m = l[0];
        for (int k = 1; k < K; ++k) m = fmax(m, l[k]);
        double s = 0.0;
        for (int k = 0; k < K; ++k) s += exp(l[k] - m);
        double lse = m + log(s);
        for (int k = 0; k < K; ++k) log_pi[(long)h * K + k] = l[k] - lse;
    }
}

/* S1 for one routing vector x[d]: gamma[k] = pi_k N(x; mu_k, diag var_k) / sum_j (...).
 * Evaluated in the log domain; ll[K] is scratch. */
static void posterior(int d, int K, const double *mu, const double *var, const double *log_pi,
                      const double *x, double *gamma, double *ll)
{
    double m = -INFINITY;
    for (int k = 0; k < K; ++k) {
        const double *mk = mu + (long)k * d, *vk = var + (long)k * d;
        double q = 0.0;
        for (int j = 0; j < d; ++j) {
            double t = x[j] - mk[j];
            q += t * t / vk[j] + log(vk[j]) + kLog2Pi;
        }
        ll[k] = log_pi[k] - 0.5 * q; /* log pi_k + log N(x; mu_k, Sigma_k) */
        m = fmax(m, ll[k]);
    }
    double den = 0.0;
    for (int k = 0; k < K; ++k) {
        gamma[k] = exp(ll[k] - m);
        den += gamma[k];
    }
    for (int k = 0; k < K; ++k) gamma[k] /= den;
}

typedef struct {
    double *var, *log_pi;
} prepared;

static prepared prepare(int H, int K, int d, const double *var_raw, const double *logit_pi)
{
    prepared p;
    p.var = (double *)malloc(sizeof(double) * (size_t)H * K * d);
    p.log_pi = (double *)malloc(sizeof(double) * (size_t)H * K);
    gma_oracle_params(H, K, d, var_raw, logit_pi, p.var, p.log_pi);
    return p;
}

static void release(prepared p)
{
    free(p.var);
    free(p.log_pi);
}

/* S1: responsibilities of S slices, gamma[s][n][K]. */
void gma_oracle_responsibilities(int S, const int *head, int H, int N, int d, int K,
                                 const double *mu, const double *var_raw, const double *logit_pi,
                                 const double *x, double *gamma)
{
    prepared p = prepare(H, K, d, var_raw, logit_pi);
#pragma omp parallel
    {
        double *ll = (double *)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(dynamic) collapse(2)
        for (int s = 0; s < S; ++s)
            for (int i = 0; i < N; ++i) {
                int h = head[s];
                posterior(d, K, mu + (long)h * K * d, p.var + (long)h * K * d, p.log_pi + (long)h * K,
                          x + ((long)s * N + i) * d, gamma + ((long)s * N + i) * K, ll);
            }
        free(ll);
    }
    release(p);
}

/* S3 for one query row: out[c] = (gq . Vt[:, c]) / (gq . Z + eps). */
static void read_row(int K, int dv, const double *gq, const double *Vt, const double *Z, double eps,
                     double *out)
{
    double den = 0.0;
    for (int k = 0; k < K; ++k) den += gq[k] * Z[k];
    den += eps;
    for (int c = 0; c < dv; ++c) {
        double num = 0.0;
        for (int k = 0; k < K; ++k) num += gq[k] * Vt[(long)k * dv + c];
        out[c] = num / den;
    }
}

/* S2 for one key row: Vt += gk v^T, Z += gk. */
static void write_row(int K, int dv, const double *gk, const double *v, double *Vt, double *Z)
{
    for (int k = 0; k < K; ++k) {
        for (int c = 0; c < dv; ++c) Vt[(long)k * dv + c] += gk[k] * v[c];
        Z[k] += gk[k];
    }
}

/* S2 alone: state[s] += [Gamma_K^T V, Gamma_K^T 1] over the slice's n key/value rows. */
void gma_oracle_write(int S, const int *head, int H, int N, int d, int dv, int K,
                      const double *mu, const double *var_raw, const double *logit_pi,
                      const double *kx, const double *v, double *state)
{
    prepared p = prepare(H, K, d, var_raw, logit_pi);
    const long sz = (long)K * dv + K;
#pragma omp parallel for schedule(dynamic)
    for (int s = 0; s < S; ++s) {
        int h = head[s];
        double *g = (double *)malloc(sizeof(double) * (size_t)K);
        double *ll = (double *)malloc(sizeof(double) * (size_t)K);
        for (int j = 0; j < N; ++j) {
            posterior(d, K, mu + (long)h * K * d, p.var + (long)h * K * d, p.log_pi + (long)h * K,
                      kx + ((long)s * N + j) * d, g, ll);
            write_row(K, dv, g, v + ((long)s * N + j) * dv, state + s * sz, state + s * sz + (long)K * dv);
        }
        free(g); free(ll);
    }
    release(p);
}

/* S3 alone: every query row of the slice reads the fixed memory state[s]. */
void gma_oracle_read(int S, const int *head, int H, int N, int d, int dv, int K,
                     const double *mu, const double *var_raw, const double *logit_pi,
                     const double *qx, const double *state, double eps, double *out)
{
    prepared p = prepare(H, K, d, var_raw, logit_pi);
    const long sz = (long)K * dv + K;
#pragma omp parallel for schedule(dynamic)
    for (int s = 0; s < S; ++s) {
        int h = head[s];
        double *g = (double *)malloc(sizeof(double) * (size_t)K);
        double *ll = (double *)malloc(sizeof(double) * (size_t)K);
        for (int i = 0; i < N; ++i) {
            posterior(d, K, mu + (long)h * K * d, p.var + (long)h * K * d, p.log_pi + (long)h * K,
                      qx + ((long)s * N + i) * d, g, ll);
            read_row(K, dv, g, state + s * sz, state + s * sz + (long)K * dv, eps,
                     out + ((long)s * N + i) * dv);
        }
        free(g); free(ll);
    }
    release(p);
}

/* S2 + S3, bidirectional: every query reads the memory written by all N keys. */
void gma_oracle_bidir(int S, const int *head, int H, int N, int d, int dv, int K,
                      const double *mu, const double *var_raw, const double *logit_pi,
                      const double *qx, const double *kx, const double *v, double eps, double *out)
{
    prepared p = prepare(H, K, d, var_raw, logit_pi);
#pragma omp parallel for schedule(dynamic)
    for (int s = 0; s < S; ++s) {
        int h = head[s];
        const double *mu_h = mu + (long)h * K * d, *var_h = p.var + (long)h * K * d;
        const double *lp_h = p.log_pi + (long)h * K;
        double *Vt = (double *)calloc((size_t)K * dv, sizeof(double));
        double *Z = (double *)calloc((size_t)K, sizeof(double));
        double *g = (double *)malloc(sizeof(double) * (size_t)K);
        double *ll = (double *)malloc(sizeof(double) * (size_t)K);
        for (int j = 0; j < N; ++j) {
            posterior(d, K, mu_h, var_h, lp_h, kx + ((long)s * N + j) * d, g, ll);
            write_row(K, dv, g, v + ((long)s * N + j) * dv, Vt, Z);
        }
        for (int i = 0; i < N; ++i) {
            posterior(d, K, mu_h, var_h, lp_h, qx + ((long)s * N + i) * d, g, ll);
            read_row(K, dv, g, Vt, Z, eps, out + ((long)s * N + i) * dv);
        }
        free(Vt); free(Z); free(g); free(ll);
    }
    release(p);
}

/* S4, causal: token i writes its key into the running memory, then its query
 * reads it, so O_i depends on tokens j <= i only.  state_in (nullable) is the
 * memory left by earlier tokens; state_out (nullable) receives the final one. */
void gma_oracle_causal(int S, const int *head, int H, int N, int d, int dv, int K,
                       const double *mu, const double *var_raw, const double *logit_pi,
                       const double *qx, const double *kx, const double *v, double eps,
                       const double *state_in, double *state_out, double *out)
{
    prepared p = prepare(H, K, d, var_raw, logit_pi);
    const long sz = (long)K * dv + K;
#pragma omp parallel for schedule(dynamic)
    for (int s = 0; s < S; ++s) {
        int h = head[s];
        const double *mu_h = mu + (long)h * K * d, *var_h = p.var + (long)h * K * d;
        const double *lp_h = p.log_pi + (long)h * K;
        double *st = (double *)calloc((size_t)sz, sizeof(double));
        if (state_in) memcpy(st, state_in + s * sz, sizeof(double) * (size_t)sz);
        double *Vt = st, *Z = st + (long)K * dv;
        double *g = (double *)malloc(sizeof(double) * (size_t)K);
        double *ll = (double *)malloc(sizeof(double) * (size_t)K);
        for (int i = 0; i < N; ++i) {
            posterior(d, K, mu_h, var_h, lp_h, kx + ((long)s * N + i) * d, g, ll);
            write_row(K, dv, g, v + ((long)s * N + i) * dv, Vt, Z);
            posterior(d, K, mu_h, var_h, lp_h, qx + ((long)s * N + i) * d, g, ll);
            read_row(K, dv, g, Vt, Z, eps, out + ((long)s * N + i) * dv);
        }
        if (state_out) memcpy(state_out + s * sz, st, sizeof(double) * (size_t)sz);
        free(st); free(g); free(ll);
    }
    release(p);
}

/* S5: one decode step per slice; state[s] is advanced in place. */
void gma_oracle_decode_step(int S, const int *head, int H, int d, int dv, int K,
                            const double *mu, const double *var_raw, const double *logit_pi,
                            const double *qx, const double *kx, const double *v, double eps,
                            double *state, double *out)
{
    gma_oracle_causal(S, head, H, 1, d, dv, K, mu, var_raw, logit_pi, qx, kx, v, eps,
                      state, state, out);
}

/* X: cross-attention.  Every query row of slice s (Nq of them) reads the
 * memory written by all Nk key/value rows of the same slice. */
void gma_oracle_cross(int S, const int *head, int H, int Nq, int Nk, int d, int dv, int K,
                      const double *mu, const double *var_raw, const double *logit_pi,
                      const double *qx, const double *kx, const double *v, double eps, double *out)
{
    prepared p = prepare(H, K, d, var_raw, logit_pi);
#pragma omp parallel for schedule(dynamic)
    for (int s = 0; s < S; ++s) {
        int h = head[s];
        const double *mu_h = mu + (long)h * K * d, *var_h = p.var + (long)h * K * d;
        const double *lp_h = p.log_pi + (long)h * K;
        double *Vt = (double *)calloc((size_t)K * dv, sizeof(double));
        double *Z = (double *)calloc((size_t)K, sizeof(double));
        double *g = (double *)malloc(sizeof(double) * (size_t)K);
        double *ll = (double *)malloc(sizeof(double) * (size_t)K);
        for (int j = 0; j < Nk; ++j) {
            posterior(d, K, mu_h, var_h, lp_h, kx + ((long)s * Nk + j) * d, g, ll);
            write_row(K, dv, g, v + ((long)s * Nk + j) * dv, Vt, Z);
        }
        for (int i = 0; i < Nq; ++i) {
            posterior(d, K, mu_h, var_h, lp_h, qx + ((long)s * Nq + i) * d, g, ll);
            read_row(K, dv, g, Vt, Z, eps, out + ((long)s * Nq + i) * dv);
        }
        free(Vt); free(Z); free(g); free(ll);
    }
    release(p);
}

/* Entropy of the distribution proportional to w[0..K-1] (w >= 0), divided by
 * log K (0 for K = 1 or an all-zero w); 0 log 0 = 0. */
static double normalised_entropy(int K, const double *w)
{
    double tot = 0.0, h = 0.0;
    for (int k = 0; k < K; ++k) tot += w[k];
    if (K < 2 || tot <= 0.0) return 0.0;
    for (int k = 0; k < K; ++k)
        if (w[k] > 0.0) {
            double q = w[k] / tot;
            h -= q * log(q);
        }
    return h / log((double)K);
}

/* D: responsibility diagnostics over the N routing rows of every slice,
 * accumulated per head (slices of the same head add up):
 *   usage[h][k]   = sum over rows of gamma_ik          (soft usage)
 *   counts[h][k]  = number of rows whose argmax is k    (hard assignments)
 *   assign[s][i]  = argmax_k gamma_ik (lowest k on ties; nullable)
 *   entropy[h][0] = normalised entropy of usage[h], entropy[h][1] of counts[h]
 * The slices of a head run one after another (no parallel sum), so the
 * result does not depend on the thread count. */
void gma_oracle_usage(int S, const int *head, int H, int N, int d, int K,
                      const double *mu, const double *var_raw, const double *logit_pi,
                      const double *x, double *usage, long long *counts, int *assign, double *entropy)
{
    prepared p = prepare(H, K, d, var_raw, logit_pi);
    for (long i = 0; i < (long)H * K; ++i) {
        usage[i] = 0.0;
        counts[i] = 0;
    }
    /* heads are independent: one thread per head, its slices in order */
#pragma omp parallel for schedule(dynamic)
    for (int h = 0; h < H; ++h) {
        double *g = (double *)malloc(sizeof(double) * (size_t)K);
        double *ll = (double *)malloc(sizeof(double) * (size_t)K);
        double *w = (double *)malloc(sizeof(double) * (size_t)K);
        for (int s = 0; s < S; ++s) {
            if (head[s] != h) continue;
            for (int i = 0; i < N; ++i) {
                posterior(d, K, mu + (long)h * K * d, p.var + (long)h * K * d, p.log_pi + (long)h * K,
                          x + ((long)s * N + i) * d, g, ll);
                int best = 0;
                for (int k = 0; k < K; ++k) {
                    usage[(long)h * K + k] += g[k];
                    if (g[k] > g[best]) best = k;
                }
                counts[(long)h * K + best] += 1;
                if (assign) assign[(long)s * N + i] = best;
            }
        }
        entropy[2 * h] = normalised_entropy(K, usage + (long)h * K);
        for (int k = 0; k < K; ++k) w[k] = (double)counts[(long)h * K + k];
        entropy[2 * h + 1] = normalised_entropy(K, w);
        free(g); free(ll); free(w);
    }
    release(p);
}

/* G: gradients of the causal (causal = 1) or bidirectional (causal = 0) form.
 *
 * With U_i = gq_i S_i ([numerator | denominator - eps]), o_i = U_i[:dv] / den_i
 * and g_i = dL/do_i:
 *   u_i          = dL/dU_i = [g_i / den_i | -(g_i . o_i) / den_i]
 *   dL/dgq_i     = S_i u_i                     (S_i: the memory row i reads)
 *   R_j          = sum over the rows i that read key j of gq_i (x) u_i
 *   dL/dgk_j     = R_j [v_j | 1],   dL/dv_j = (gk_j R_j)[:dv]
 * (causal: S_i = sum_{j <= i}, R_j = sum_{i >= j}; bidirectional: all rows).
 * Through the softmax over components, delta_ik = gamma_ik (dL/dgamma_ik -
 * sum_k' gamma_ik' dL/dgamma_ik'), and through the log-joint
 *   l_ik = log pi_k - 1/2 sum_d [(x_id - mu_kd)^2 / s_kd + log s_kd + log 2 pi],
 * s = sigma^2:
 *   dL/dx_id   = -sum_k delta_ik (x_id - mu_kd) / s_kd
 *   dL/dmu_kd += delta_ik (x_id - mu_kd) / s_kd
 *   dL/ds_kd  += delta_ik (1/2 (x_id - mu_kd)^2 / s_kd^2 - 1/2 / s_kd)
 *   dL/dlogpi_k += delta_ik
 * over the query and key rows of every slice of the head; finally
 *   dL/dvar_raw = dL/ds * sigmoid(var_raw)      (softplus' = sigmoid)
 *   dL/dlogit_k = G_k - pi_k sum_k' G_k'        (log-softmax), G = dL/dlogpi.
 * Outputs dqx, dkx [S][N][d], dv [S][N][dv]; dmu, dvar_raw [H][K][d] and
 * dlogit [H][K] are overwritten (the sum over the slices of each head, taken
 * in slice order). */
void gma_oracle_backward(int S, const int *head, int H, int N, int d, int dv, int K, int causal,
                         const double *mu, const double *var_raw, const double *logit_pi,
                         const double *qx, const double *kx, const double *v, double eps,
                         const double *dout, double *dqx, double *dkx, double *dv_out,
                         double *dmu, double *dvar_raw, double *dlogit)
{
    prepared p = prepare(H, K, d, var_raw, logit_pi);
    const long w = (long)dv + 1, kd = (long)K * d;
    /* per-slice parameter gradients, summed in slice order after the parallel loop */
    double *pmu = (double *)calloc((size_t)S * kd, sizeof(double));
    double *pvar = (double *)calloc((size_t)S * kd, sizeof(double));
    double *plp = (double *)calloc((size_t)S * K, sizeof(double));
#pragma omp parallel for schedule(dynamic)
    for (int s = 0; s < S; ++s) {
        int h = head[s];
        const double *mu_h = mu + (long)h * kd, *var_h = p.var + (long)h * kd;
        const double *lp_h = p.log_pi + (long)h * K;
        const double *xq = qx + (long)s * N * d, *xk = kx + (long)s * N * d;
        const double *vs = v + (long)s * N * dv, *gs = dout + (long)s * N * dv;
        double *gq = (double *)malloc(sizeof(double) * (size_t)N * K);
        double *gk = (double *)malloc(sizeof(double) * (size_t)N * K);
        double *dgq = (double *)malloc(sizeof(double) * (size_t)N * K);
        double *dgk = (double *)malloc(sizeof(double) * (size_t)N * K);
        double *u = (double *)malloc(sizeof(double) * (size_t)N * w);
        double *M = (double *)calloc((size_t)K * w, sizeof(double));   /* S_i, then R_j */
        double *ll = (double *)malloc(sizeof(double) * (size_t)K);
        double *vrow = (double *)malloc(sizeof(double) * (size_t)w);
        for (int i = 0; i < N; ++i) {
            posterior(d, K, mu_h, var_h, lp_h, xq + (long)i * d, gq + (long)i * K, ll);
            posterior(d, K, mu_h, var_h, lp_h, xk + (long)i * d, gk + (long)i * K, ll);
        }
        /* the write: S accumulates gk_j (x) [v_j | 1]; bidirectional: all of it first */
        if (!causal)
            for (int j = 0; j < N; ++j)
                for (int k = 0; k < K; ++k) {
                    for (int c = 0; c < dv; ++c) M[k * w + c] += gk[(long)j * K + k] * vs[(long)j * dv + c];
                    M[k * w + dv] += gk[(long)j * K + k];
                }
        for (int i = 0; i < N; ++i) {
            if (causal)
                for (int k = 0; k < K; ++k) {
                    for (int c = 0; c < dv; ++c) M[k * w + c] += gk[(long)i * K + k] * vs[(long)i * dv + c];
                    M[k * w + dv] += gk[(long)i * K + k];
                }
            /* the read of row i, then u_i and dL/dgq_i */
            double den = eps, go = 0.0;
            for (int k = 0; k < K; ++k) den += gq[(long)i * K + k] * M[k * w + dv];
            for (int c = 0; c < dv; ++c) {
                double num = 0.0;
                for (int k = 0; k < K; ++k) num += gq[(long)i * K + k] * M[k * w + c];
                go += gs[(long)i * dv + c] * (num / den);
            }
            double *ui = u + (long)i * w;
            for (int c = 0; c < dv; ++c) ui[c] = gs[(long)i * dv + c] / den;
            ui[dv] = -go / den;
            for (int k = 0; k < K; ++k) {
                double t = 0.0;
                for (int c = 0; c < w; ++c) t += M[k * w + c] * ui[c];
                dgq[(long)i * K + k] = t;
            }
        }
        /* R: the rows that read key j; causal: i >= j (a suffix, inclusive) */
        for (long e = 0; e < (long)K * w; ++e) M[e] = 0.0;
        if (!causal)
            for (int i = 0; i < N; ++i)
                for (int k = 0; k < K; ++k)
                    for (int c = 0; c < w; ++c) M[k * w + c] += gq[(long)i * K + k] * u[(long)i * w + c];
        for (int j = N - 1; j >= 0; --j) {
            if (causal)
                for (int k = 0; k < K; ++k)
                    for (int c = 0; c < w; ++c) M[k * w + c] += gq[(long)j * K + k] * u[(long)j * w + c];
            for (int c = 0; c < dv; ++c) vrow[c] = vs[(long)j * dv + c];
            vrow[dv] = 1.0;
            for (int k = 0; k < K; ++k) {
                double t = 0.0;
                for (int c = 0; c < w; ++c) t += M[k * w + c] * vrow[c];
                dgk[(long)j * K + k] = t;
            }
            for (int c = 0; c < dv; ++c) {
                double t = 0.0;
                for (int k = 0; k < K; ++k) t += gk[(long)j * K + k] * M[k * w + c];
                dv_out[((long)s * N + j) * dv + c] = t;
            }
        }
        /* through the softmax and the log-joint, for the query rows then the key rows */
        for (int pass = 0; pass < 2; ++pass) {
            const double *x = pass ? xk : xq, *g = pass ? gk : gq, *dg = pass ? dgk : dgq;
            double *dx = (pass ? dkx : dqx) + (long)s * N * d;
            for (int i = 0; i < N; ++i) {
                double dot = 0.0;
                for (int k = 0; k < K; ++k) dot += g[(long)i * K + k] * dg[(long)i * K + k];
                for (int j2 = 0; j2 < d; ++j2) dx[(long)i * d + j2] = 0.0;
                for (int k = 0; k < K; ++k) {
                    const double delta = g[(long)i * K + k] * (dg[(long)i * K + k] - dot);
                    plp[(long)s * K + k] += delta;
                    for (int j2 = 0; j2 < d; ++j2) {
                        const double t = x[(long)i * d + j2] - mu_h[(long)k * d + j2], sk = var_h[(long)k * d + j2];
                        dx[(long)i * d + j2] -= delta * t / sk;
                        pmu[(long)s * kd + (long)k * d + j2] += delta * t / sk;
                        pvar[(long)s * kd + (long)k * d + j2] += delta * (0.5 * t * t / (sk * sk) - 0.5 / sk);
                    }
                }
            }
        }
        free(gq); free(gk); free(dgq); free(dgk); free(u); free(M); free(ll); free(vrow);
    }
    for (long e = 0; e < (long)H * kd; ++e) {
        dmu[e] = 0.0;
        dvar_raw[e] = 0.0;
    }
    for (long e = 0; e < (long)H * K; ++e) dlogit[e] = 0.0;
    for (int s = 0; s < S; ++s) {
        int h = head[s];
        for (long e = 0; e < kd; ++e) {
            dmu[(long)h * kd + e] += pmu[(long)s * kd + e];
            dvar_raw[(long)h * kd + e] += pvar[(long)s * kd + e];
        }
        for (int k = 0; k < K; ++k) dlogit[(long)h * K + k] += plp[(long)s * K + k];
    }
    for (long e = 0; e < (long)H * kd; ++e) dvar_raw[e] *= 1.0 / (1.0 + exp(-var_raw[e]));
    for (int h = 0; h < H; ++h) {
        double tot = 0.0;
        for (int k = 0; k < K; ++k) tot += dlogit[(long)h * K + k];
        for (int k = 0; k < K; ++k) dlogit[(long)h * K + k] -= exp(p.log_pi[(long)h * K + k]) * tot;
    }
    free(pmu); free(pvar); free(plp);
    release(p);
}
