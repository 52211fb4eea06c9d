/*
 * Falcon fast-weight forward pass: the fp64 token-by-token recurrence (the oracle).
 *
 * TEST INFRASTRUCTURE. This file is the reference the CUDA path is checked
 * against. Only the tests, the smoke check and the benchmark's CPU-baseline leg
 * may load it. It shares no code, header, table or helper with the CUDA path.
 *
 * Sources ("Fast Weight Attention for Continual Learning", arXiv 2608.27763, as
 * summarised on three web pages):
 *   [PL]  paperlayer.ai source-linked summary (sections as it labels them)
 *   [AH]  agihunt.info explainer "Falcon realigns fast-weight writes"
 *   [SG]  sungsoo.github.io post on Falcon (Korean)
 *
 * What is computed, per (batch, head) sequence, for global steps
 * tau = pos+1 .. pos+T (one step per input token):
 *   prefix-aligned pair   x_tau = phi(k_{tau-1}), y_tau = v_tau, phi = identity,
 *                         sentinel x_1 = 0                [PL abstract; PL §3; PL Appendix p.34;
 *                                                           PL §H.3 "unkernelized case"]
 *   NLMS step             eta = beta / (||x||^2 + lambda + eps), eta = 0 when the
 *                         denominator is 0                 [PL §3.1; PL Appendix p.34; AH Method]
 *   ridge decay           alpha = min(eta*lambda, 1 - eps_gamma), gamma = 1 - alpha,
 *                         and eta_1 = alpha_1 = 0, gamma_1 = 1 at tau = 1
 *                                                          [PL §C.3; PL §4.6; SG ridge paragraph]
 *   Falcon-1              r = y - S_{tau-1}^T x,  S = gamma S + eta x r^T
 *                                                          [AH Method; SG pre-update residual]
 *   Falcon-1A             S = gamma S + eta x y^T          [AH Method "the A family writes"]
 *   Falcon-2              per value column c: eta_c = beta_c/den, gamma_c from eta_c,
 *                         column c follows the Falcon-1 rule with its own scalars
 *                                                          [PL §1 "Falcon-2"; PL Figure 5 / Parallel Form]
 *   Falcon-3              window I = {j : max(2, tau-W+1) <= j <= tau}, B = |I|;
 *                         mu = lambda_max((1/B) sum_{j in I} x_j x_j^T);
 *                         eta = beta/(mu + lambda + eps); residuals r_j = y_j - S_{tau-1}^T x_j
 *                         for every j in I (all at the pre-update state);
 *                         S = gamma S + (eta/B) sum_j x_j r_j^T
 *                                                          [PL §4.4; PL §C.6 "exact top eigenvalue";
 *                                                           AH Method; SG step-size paragraph]
 *   Falcon-2A             per value column c, the Falcon-1A write with eta_c = beta_c/den and
 *                         gamma_c from eta_c: S[:,c] = gamma_c S[:,c] + eta_c x y_c
 *                                                          [PL §4.3 "the A family"; PL "B. Falcon-2A"]
 *   Falcon-3A             the Falcon-3 window, written with the targets themselves:
 *                         E = (1/B) sum_{j in I} ||x_j||^2 (the window's mean key energy),
 *                         eta = beta/(E + lambda + eps), S = gamma S + (eta/B) sum_j x_j y_j^T
 *                                                          [PL §4.3; PL §4.5; PL §4.6; PL "C. Falcon-3A"]
 *   read                  o_tau = S_tau^T q_tau (read after write)  [AH Method; SG RAW paragraph]
 *   continuation tail     the last W keys and last W-1 values, so that the next
 *                         segment's first pair and window are exact  [PL §C.7; PL §4.4]
 *
 * Readings where the pages are silent or garbled (each is also listed in the
 * design notes): the residual uses S_{tau-1} (PL "A More on Background" prints
 * S_t, which contradicts PL §4.4, AH and SG); the sentinel pair j = 1 is not a
 * member of the Falcon-3 window (PL §4.5 "skips the boundary update at t = 1");
 * Falcon-2 shares the denominator ||x||^2 + lambda + eps across columns and
 * only beta is per column (so does Falcon-2A); the tail also carries the pending key k_T; the
 * pages normalise Falcon-3A's step by the "window energy" without printing it: read here as the
 * mean of ||x_j||^2 over the window, which keeps W = 1 equal to Falcon-1A and does not grow with W.
 *
 * Arithmetic: plain fp64, token by token, no reassociation tricks. Compile
 * without -ffast-math.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define REF_F1 1
#define REF_F1A 2
#define REF_F2 3
#define REF_F2A 4
#define REF_F3 5
#define REF_F3A 6

#define REF_OK 0
#define REF_EINVAL 1
#define REF_ENOMEM 2

/* Largest eigenvalue of a symmetric n x n matrix (row-major, overwritten), by
 * cyclic Jacobi rotations in fp64 (the classical method: each rotation zeroes one
 * off-diagonal pair; sweeps repeat until the off-diagonal mass is negligible). */
static double jacobi_lambda_max(int n, double *a) {
    for (int sweep = 0; sweep < 100; ++sweep) {
        double off = 0.0, diag = 0.0;
        for (int p = 0; p < n; ++p) {
            diag += a[p * n + p] * a[p * n + p];
            for (int q = p + 1; q < n; ++q) off += a[p * n + q] * a[p * n + q];
        }
        if (off == 0.0 || off <= 1e-34 * diag) break;
        for (int p = 0; p < n; ++p) {
            for (int q = p + 1; q < n; ++q) {
                double apq = a[p * n + q];
                if (apq == 0.0) continue;
                double theta = (a[q * n + q] - a[p * n + p]) / (2.0 * apq);
                double t = (theta >= 0.0 ? 1.0 : -1.0) / (fabs(theta) + sqrt(theta * theta + 1.0));
                double c = 1.0 / sqrt(t * t + 1.0), s = t * c;
                for (int k = 0; k < n; ++k) { /* A <- A J */
                    double akp = a[k * n + p], akq = a[k * n + q];
                    a[k * n + p] = c * akp - s * akq;
                    a[k * n + q] = s * akp + c * akq;
                }
                for (int k = 0; k < n; ++k) { /* A <- J^T A */
                    double apk = a[p * n + k], aqk = a[q * n + k];
                    a[p * n + k] = c * apk - s * aqk;
                    a[q * n + k] = s * apk + c * aqk;
                }
            }
        }
    }
    double m = a[0];
    for (int p = 1; p < n; ++p)
        if (a[p * n + p] > m) m = a[p * n + p];
    return m;
}

/* Exported so tests can compare it with a library eigensolver. */
double falcon_ref_lambda_max(int n, const double *g) {
    if (n <= 0) return 0.0;
    double *a = (double *)malloc(sizeof(double) * (size_t)n * (size_t)n);
    if (!a) return NAN;
    memcpy(a, g, sizeof(double) * (size_t)n * (size_t)n);
    double m = jacobi_lambda_max(n, a);
    free(a);
    return m;
}

typedef struct {
    int variant, W;
    int64_t T, dk, dv, pos;
    const double *q, *k, *v;   /* [T,dk], [T,dk], [T,dv] of this sequence */
    const double *beta;        /* [T] (Falcon-2: [T,dv]) */
    const double *lam;         /* [T] */
    const double *S0;          /* [dk,dv] or NULL */
    const double *tk, *tv;     /* tail: [W,dk] keys k_{pos-W+1..pos}; [W-1,dv] values v_{pos-W+2..pos} */
    double eps, eps_gamma;
    double *out, *S, *tk_out, *tv_out;
    double *work;              /* scratch: see run_sequence */
} seq_job;

/* Key k at global index i (1-based). Indices <= 0 do not exist: zero. */
static const double *key_at(const seq_job *j, int64_t i, const double *zeros) {
    if (i <= 0) return zeros;
    if (i <= j->pos) return j->tk + (i - (j->pos - j->W + 1)) * j->dk;
    return j->k + (i - j->pos - 1) * j->dk;
}

static const double *val_at(const seq_job *j, int64_t i, const double *zeros) {
    if (i <= 0) return zeros;
    if (i <= j->pos) return j->tv + (i - (j->pos - j->W + 2)) * j->dv;
    return j->v + (i - j->pos - 1) * j->dv;
}

static void run_sequence(seq_job *j) {
    const int64_t dk = j->dk, dv = j->dv, W = j->W;
    double *S = j->S;
    double *zeros = j->work;           /* max(dk,dv) zeros */
    double *pred = zeros + (dk > dv ? dk : dv); /* dv: S^T x */
    double *res = pred + dv;           /* W*dv residuals */
    double *gram = res + W * dv;       /* W*W */
    const double **xs = (const double **)(gram + W * W); /* W pointers */
    const double **ys = xs + W;

    if (j->S0) memcpy(S, j->S0, sizeof(double) * dk * dv);
    else memset(S, 0, sizeof(double) * dk * dv);

    for (int64_t t = 0; t < j->T; ++t) {
        const int64_t tau = j->pos + t + 1;
        const double lam = j->lam[t];
        const double *y = j->v + t * dv;
        if (j->variant == REF_F3 || j->variant == REF_F3A) {
            int64_t jlo = tau - W + 1;
            if (jlo < 2) jlo = 2;
            const int64_t B = tau >= 2 ? tau - jlo + 1 : 0;
            if (B > 0) {
                for (int64_t a = 0; a < B; ++a) {
                    xs[a] = key_at(j, jlo + a - 1, zeros);
                    ys[a] = val_at(j, jlo + a, zeros);
                }
                for (int64_t a = 0; a < B; ++a)
                    for (int64_t b = 0; b < B; ++b) {
                        double g = 0.0;
                        for (int64_t c = 0; c < dk; ++c) g += xs[a][c] * xs[b][c];
                        gram[a * B + b] = g / (double)B;
                    }
                double mu;
                if (j->variant == REF_F3) {
                    mu = jacobi_lambda_max((int)B, gram);
                } else { /* Falcon-3A: the window's mean key energy, the trace of the averaged Gram */
                    mu = 0.0;
                    for (int64_t a = 0; a < B; ++a) mu += gram[a * B + a];
                }
                const double den = mu + lam + j->eps;
                const double eta = den == 0.0 ? 0.0 : j->beta[t] / den;
                double alpha = eta * lam;
                if (alpha > 1.0 - j->eps_gamma) alpha = 1.0 - j->eps_gamma;
                const double gamma = 1.0 - alpha;
                for (int64_t a = 0; a < B; ++a)       /* residuals at S_{tau-1} (Falcon-3A: the targets) */
                    for (int64_t c = 0; c < dv; ++c) {
                        double p = 0.0;
                        if (j->variant == REF_F3)
                            for (int64_t r = 0; r < dk; ++r) p += S[r * dv + c] * xs[a][r];
                        res[a * dv + c] = ys[a][c] - p;
                    }
                const double w = eta / (double)B;
                for (int64_t r = 0; r < dk; ++r)
                    for (int64_t c = 0; c < dv; ++c) {
                        double acc = 0.0;
                        for (int64_t a = 0; a < B; ++a) acc += xs[a][r] * res[a * dv + c];
                        S[r * dv + c] = gamma * S[r * dv + c] + w * acc;
                    }
            }
        } else if (tau >= 2) { /* tau == 1: x = 0, eta = alpha = 0, gamma = 1: no-op */
            const double *x = key_at(j, tau - 1, zeros);
            double nx = 0.0;
            for (int64_t r = 0; r < dk; ++r) nx += x[r] * x[r];
            const double den = nx + lam + j->eps;
            if (j->variant == REF_F2 || j->variant == REF_F2A) {
                const double *bt = j->beta + t * dv;
                for (int64_t c = 0; c < dv; ++c) {
                    const double eta = den == 0.0 ? 0.0 : bt[c] / den;
                    double alpha = eta * lam;
                    if (alpha > 1.0 - j->eps_gamma) alpha = 1.0 - j->eps_gamma;
                    const double gamma = 1.0 - alpha;
                    double p = 0.0; /* Falcon-2A writes the target itself */
                    if (j->variant == REF_F2)
                        for (int64_t r = 0; r < dk; ++r) p += S[r * dv + c] * x[r];
                    const double rc = y[c] - p;
                    for (int64_t r = 0; r < dk; ++r) S[r * dv + c] = gamma * S[r * dv + c] + eta * x[r] * rc;
                }
            } else {
                const double eta = den == 0.0 ? 0.0 : j->beta[t] / den;
                double alpha = eta * lam;
                if (alpha > 1.0 - j->eps_gamma) alpha = 1.0 - j->eps_gamma;
                const double gamma = 1.0 - alpha;
                if (j->variant == REF_F1) {
                    for (int64_t c = 0; c < dv; ++c) {
                        double p = 0.0;
                        for (int64_t r = 0; r < dk; ++r) p += S[r * dv + c] * x[r];
                        pred[c] = y[c] - p; /* residual at S_{tau-1} */
                    }
                    for (int64_t r = 0; r < dk; ++r)
                        for (int64_t c = 0; c < dv; ++c) S[r * dv + c] = gamma * S[r * dv + c] + eta * x[r] * pred[c];
                } else { /* Falcon-1A: inner-product write of the target itself */
                    for (int64_t r = 0; r < dk; ++r)
                        for (int64_t c = 0; c < dv; ++c) S[r * dv + c] = gamma * S[r * dv + c] + eta * x[r] * y[c];
                }
            }
        }
        /* read after write */
        const double *qt = j->q + t * dk;
        double *o = j->out + t * dv;
        for (int64_t c = 0; c < dv; ++c) {
            double acc = 0.0;
            for (int64_t r = 0; r < dk; ++r) acc += S[r * dv + c] * qt[r];
            o[c] = acc;
        }
    }
    const int64_t end = j->pos + j->T;
    for (int64_t a = 0; a < W; ++a) {
        const double *kk = key_at(j, end - W + 1 + a, zeros);
        memcpy(j->tk_out + a * dk, kk, sizeof(double) * dk);
    }
    for (int64_t a = 0; a + 1 < W; ++a) {
        const double *vv = val_at(j, end - W + 2 + a, zeros);
        memcpy(j->tv_out + a * dv, vv, sizeof(double) * dv);
    }
}

typedef struct {
    seq_job *jobs;
    int64_t njobs;
    int64_t next;
    pthread_mutex_t mu;
} pool_t;

static void *worker(void *arg) {
    pool_t *p = (pool_t *)arg;
    for (;;) {
        pthread_mutex_lock(&p->mu);
        int64_t i = p->next++;
        pthread_mutex_unlock(&p->mu);
        if (i >= p->njobs) return NULL;
        run_sequence(&p->jobs[i]);
    }
}

/*
 * Arrays are contiguous fp64 in the layouts below ([B,H,...] outermost).
 *   q, k: [B,H,T,dk]   v: [B,H,T,dv]   beta: [B,H,T] (Falcon-2: [B,H,T,dv])
 *   (Falcon-2A: [B,H,T,dv] as well)
 *   lam: [B,H,T]       S0: [B,H,dk,dv] or NULL (zero state)
 *   tail_k: [B,H,W,dk] holding k_{pos-W+1..pos}; tail_v: [B,H,W-1,dv] holding
 *   v_{pos-W+2..pos}; both NULL iff pos == 0. Entries at global index <= 0 are zero.
 *   out: [B,H,T,dv]  S_final: [B,H,dk,dv]  tail_k_out / tail_v_out: as tail_k / tail_v
 *   for position pos + T.
 * window must be 1 except for Falcon-3 and 3A. nthreads <= 0 means one thread.
 * Returns 0, or 1 for invalid arguments, 2 when memory runs out.
 */
int falcon_ref_fwd(int variant, int64_t B, int64_t H, int64_t T, int64_t dk, int64_t dv, int window,
                   int64_t pos, const double *q, const double *k, const double *v, const double *beta,
                   const double *lam, const double *S0, const double *tail_k, const double *tail_v,
                   double eps, double eps_gamma, double *out, double *S_final, double *tail_k_out,
                   double *tail_v_out, int nthreads) {
    if (variant < REF_F1 || variant > REF_F3A) return REF_EINVAL;
    if (B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0 || window < 1 || pos < 0) return REF_EINVAL;
    if (variant != REF_F3 && variant != REF_F3A && window != 1) return REF_EINVAL;
    if ((pos > 0) != (tail_k != NULL)) return REF_EINVAL;
    if (pos > 0 && window > 1 && tail_v == NULL) return REF_EINVAL;
    const int64_t n = B * H;
    if (n == 0) return REF_OK;
    const int64_t W = window;
    const int64_t wlen = (dk > dv ? dk : dv) + dv + W * dv + W * W + 2 * W + 2;
    seq_job *jobs = (seq_job *)calloc((size_t)n, sizeof(seq_job));
    double *work = (double *)calloc((size_t)(n * wlen), sizeof(double));
    if (!jobs || !work) {
        free(jobs);
        free(work);
        return REF_ENOMEM;
    }
    const int bt_stride = (variant == REF_F2 || variant == REF_F2A) ? (int)dv : 1;
    for (int64_t s = 0; s < n; ++s) {
        seq_job *j = &jobs[s];
        j->variant = variant;
        j->W = (int)W;
        j->T = T;
        j->dk = dk;
        j->dv = dv;
        j->pos = pos;
        j->q = q + s * T * dk;
        j->k = k + s * T * dk;
        j->v = v + s * T * dv;
        j->beta = beta + s * T * bt_stride;
        j->lam = lam + s * T;
        j->S0 = S0 ? S0 + s * dk * dv : NULL;
        j->tk = tail_k ? tail_k + s * W * dk : NULL;
        j->tv = tail_v ? tail_v + s * (W - 1) * dv : NULL;
        j->eps = eps;
        j->eps_gamma = eps_gamma;
        j->out = out + s * T * dv;
        j->S = S_final + s * dk * dv;
        j->tk_out = tail_k_out + s * W * dk;
        j->tv_out = tail_v_out + s * (W - 1) * dv;
        j->work = work + s * wlen;
    }
    if (nthreads <= 1) {
        for (int64_t s = 0; s < n; ++s) run_sequence(&jobs[s]);
    } else {
        if (nthreads > n) nthreads = (int)n;
        pool_t p;
        p.jobs = jobs;
        p.njobs = n;
        p.next = 0;
        pthread_mutex_init(&p.mu, NULL);
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        int started = 0;
        for (int i = 0; th && i < nthreads; ++i)
            if (pthread_create(&th[i], NULL, worker, &p) == 0) ++started;
        if (started == 0) worker(&p);
        for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
        free(th);
        pthread_mutex_destroy(&p.mu);
    }
    free(jobs);
    free(work);
    return REF_OK;
}
