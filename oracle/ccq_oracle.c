/*
 * ccq_oracle.c -- plain fp64 CPU oracle for the CCQ linear-attention forward.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load or call this code.  It shares nothing with the
 * CUDA library: no header, no helper, no constant.
 *
 * What it computes, token by token, for every (batch, head) pair, exactly as
 * the CCQ pages define it:
 *
 *   backbone write (unchanged by CCQ; gist.science summary of 2606.01294,
 *   section 2 "integration": S_t = Update(S_{t-1}; k_t, v_t, ...)):
 *     GLA  : S_t = Diag(alpha_t) S_{t-1} + k_t v_t^T          alpha_t per channel
 *     GDN  : S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *   key statistics (same summary, section 2 "mechanism": one extra d_k x d_k
 *   matrix and one d_k vector per head; the 10100.com article, "cost and
 *   limits": the covariance is undecayed):
 *     C_t = C_{t-1} + k_t k_t^T,  m_t = m_{t-1} + k_t,  n_t = n_{t-1} + 1
 *   curvature (same summary, section 2 "theory": the Hessian at q = 0 of
 *   A_t(q) = log sum_{j<=t} exp(k_j^T q) is the running key covariance):
 *     Sigma_t = C_t / n_t - (m_t / n_t)(m_t / n_t)^T
 *   read (10100.com article "method", item 1; summary section 2):
 *     lambda_t = sigmoid(w_lambda[h] . q_t + b_lambda[h])   (or a given lambda)
 *     q_clean  = q_t - lambda_t Sigma_t q_t
 *     o_t      = S_t^T q_clean            (S is d_k x d_v; the page writes S q)
 *
 * Readings where the pages are silent (all listed in the design notes):
 *   - the read uses S_t after the write of token t, and Sigma_t includes k_t;
 *   - n counts every token seen, including a carried prefix (t0);
 *   - Sigma is the population covariance (divide by n, not n-1): it is the
 *     Hessian of log-sum-exp at q = 0 with uniform softmax weights 1/n;
 *   - with the l2norm switch, q and k are first scaled by 1/sqrt(|x|^2+1e-6)
 *     and that normalised q feeds both the gate and the read.
 *
 * All arithmetic is fp64.  Threads split the (b, h) pairs; each pair is a
 * strictly sequential loop over tokens, so the result does not depend on the
 * thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int backbone; /* 0 = GLA, 1 = Gated DeltaNet */
    const double *q, *k, *v, *log_alpha, *beta;
    const double *w_lambda, *b_lambda, *lambda_in;
    int l2norm;
    const double *S0, *C0, *m0;
    int64_t t0;
    double *o, *lambda_out, *sigq_out, *S_out, *C_out, *m_out;
    int B, H, T, dk, dv;
    int next_pair; /* work counter, guarded by mu */
    pthread_mutex_t mu;
    int status;
} job_t;

static void normalise(double *x, int d)
{
    double ss = 0.0;
    for (int i = 0; i < d; ++i) ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss + 1e-6);
    for (int i = 0; i < d; ++i) x[i] *= r;
}

static int run_pair(const job_t *J, int bh, double *work)
{
    const int dk = J->dk, dv = J->dv, T = J->T, h = bh % J->H;
    double *S = work;                 /* dk x dv */
    double *C = S + (size_t)dk * dv;  /* dk x dk */
    double *m = C + (size_t)dk * dk;  /* dk */
    double *q = m + dk, *k = q + dk, *v = k + dk; /* v: dv */
    double *Cq = v + dv, *kS = Cq + dk, *qc = kS + dv; /* kS: dv */

    if (J->S0) memcpy(S, J->S0 + (size_t)bh * dk * dv, sizeof(double) * dk * dv);
    else memset(S, 0, sizeof(double) * dk * dv);
    if (J->C0) memcpy(C, J->C0 + (size_t)bh * dk * dk, sizeof(double) * dk * dk);
    else memset(C, 0, sizeof(double) * dk * dk);
    if (J->m0) memcpy(m, J->m0 + (size_t)bh * dk, sizeof(double) * dk);
    else memset(m, 0, sizeof(double) * dk);
    double n = (double)J->t0;

    for (int t = 0; t < T; ++t) {
        size_t tok = (size_t)bh * T + t;
        memcpy(q, J->q + tok * dk, sizeof(double) * dk);
        memcpy(k, J->k + tok * dk, sizeof(double) * dk);
        memcpy(v, J->v + tok * dv, sizeof(double) * dv);
        if (J->l2norm) {
            normalise(q, dk);
            normalise(k, dk);
        }

        /* backbone write */
        if (J->backbone == 0) {
            const double *la = J->log_alpha + tok * dk;
            for (int i = 0; i < dk; ++i) {
                double a = exp(la[i]);
                double *Si = S + (size_t)i * dv;
                for (int j = 0; j < dv; ++j) Si[j] = a * Si[j] + k[i] * v[j];
            }
        } else {
            double a = exp(J->log_alpha[tok]);
            double b = J->beta[tok];
            for (int j = 0; j < dv; ++j) kS[j] = 0.0;
            for (int i = 0; i < dk; ++i) {
                const double *Si = S + (size_t)i * dv;
                for (int j = 0; j < dv; ++j) kS[j] += k[i] * Si[j];
            }
            for (int i = 0; i < dk; ++i) {
                double *Si = S + (size_t)i * dv;
                for (int j = 0; j < dv; ++j)
                    Si[j] = a * (Si[j] - b * k[i] * kS[j]) + b * k[i] * v[j];
            }
        }

        /* undecayed key statistics */
        for (int i = 0; i < dk; ++i) {
            double *Ci = C + (size_t)i * dk;
            for (int j = 0; j < dk; ++j) Ci[j] += k[i] * k[j];
            m[i] += k[i];
        }
        n += 1.0;

        /* Sigma_t q = C q / n - mu (mu . q) */
        double muq = 0.0;
        for (int i = 0; i < dk; ++i) muq += (m[i] / n) * q[i];
        for (int i = 0; i < dk; ++i) {
            const double *Ci = C + (size_t)i * dk;
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += Ci[j] * q[j];
            Cq[i] = acc / n - (m[i] / n) * muq;
        }

        /* gate */
        double lam;
        if (J->lambda_in) {
            lam = J->lambda_in[tok];
        } else {
            double z = J->b_lambda[h];
            const double *w = J->w_lambda + (size_t)h * dk;
            for (int i = 0; i < dk; ++i) z += w[i] * q[i];
            lam = 1.0 / (1.0 + exp(-z));
        }
        if (J->lambda_out) J->lambda_out[tok] = lam;
        if (J->sigq_out) memcpy(J->sigq_out + tok * dk, Cq, sizeof(double) * dk);

        /* read: o_t = S_t^T q_clean */
        for (int i = 0; i < dk; ++i) qc[i] = q[i] - lam * Cq[i];
        double *o = J->o + tok * dv;
        for (int j = 0; j < dv; ++j) o[j] = 0.0;
        for (int i = 0; i < dk; ++i) {
            const double *Si = S + (size_t)i * dv;
            for (int j = 0; j < dv; ++j) o[j] += qc[i] * Si[j];
        }
    }

    if (J->S_out) memcpy(J->S_out + (size_t)bh * dk * dv, S, sizeof(double) * dk * dv);
    if (J->C_out) memcpy(J->C_out + (size_t)bh * dk * dk, C, sizeof(double) * dk * dk);
    if (J->m_out) memcpy(J->m_out + (size_t)bh * dk, m, sizeof(double) * dk);
    return 0;
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    size_t words = (size_t)J->dk * J->dv + (size_t)J->dk * J->dk + 6 * (size_t)J->dk +
                   3 * (size_t)J->dv;
    double *work = (double *)malloc(sizeof(double) * words);
    if (!work) {
        pthread_mutex_lock(&J->mu);
        J->status = 2;
        pthread_mutex_unlock(&J->mu);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int bh = J->next_pair++;
        pthread_mutex_unlock(&J->mu);
        if (bh >= J->B * J->H) break;
        run_pair(J, bh, work);
    }
    free(work);
    return NULL;
}

/*
 * Returns 0 on success, 1 on a bad argument, 2 on an allocation failure.
 * All arrays are fp64, row-major: q,k [B,H,T,dk]; v,o [B,H,T,dv];
 * log_alpha [B,H,T,dk] (GLA) or [B,H,T] (GDN); beta [B,H,T] (GDN only);
 * w_lambda [H,dk]; b_lambda [H]; lambda_in/lambda_out [B,H,T];
 * sigq_out [B,H,T,dk] (Sigma_t q_t, for checks); S [B,H,dk,dv];
 * C [B,H,dk,dk]; m [B,H,dk].  Nullable: beta (GLA), lambda_in, lambda_out,
 * sigq_out, S0/C0/m0 (all or none), S_out, C_out, m_out.
 */
int ccq_oracle_fwd(int backbone, const double *q, const double *k, const double *v,
                   const double *log_alpha, const double *beta, const double *w_lambda,
                   const double *b_lambda, const double *lambda_in, int l2norm,
                   const double *S0, const double *C0, const double *m0, int64_t t0,
                   double *o, double *lambda_out, double *sigq_out, double *S_out,
                   double *C_out, double *m_out, int B, int H, int T, int dk, int dv,
                   int nthreads)
{
    if (backbone != 0 && backbone != 1) return 1;
    if (!q || !k || !v || !log_alpha || !o || B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0)
        return 1;
    if (backbone == 1 && !beta) return 1;
    if (!lambda_in && (!w_lambda || !b_lambda)) return 1;
    int any0 = (S0 != NULL) + (C0 != NULL) + (m0 != NULL);
    if (any0 != 0 && any0 != 3) return 1;
    if (any0 == 0 && t0 != 0) return 1;
    if (t0 < 0) return 1;

    job_t J;
    memset(&J, 0, sizeof(J));
    J.backbone = backbone;
    J.q = q; J.k = k; J.v = v; J.log_alpha = log_alpha; J.beta = beta;
    J.w_lambda = w_lambda; J.b_lambda = b_lambda; J.lambda_in = lambda_in;
    J.l2norm = l2norm;
    J.S0 = S0; J.C0 = C0; J.m0 = m0; J.t0 = t0;
    J.o = o; J.lambda_out = lambda_out; J.sigq_out = sigq_out;
    J.S_out = S_out; J.C_out = C_out; J.m_out = m_out;
    J.B = B; J.H = H; J.T = T; J.dk = dk; J.dv = dv;
    pthread_mutex_init(&J.mu, NULL);

    int pairs = B * H;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > pairs) nthreads = pairs > 0 ? pairs : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) return 2;
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, worker, &J) != 0) break;
        ++started;
    }
    if (started == 0) worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.mu);
    return J.status;
}
