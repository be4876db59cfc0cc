/*
 * CPU oracle for the gated delta rule -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain token-by-token recurrence in fp64.  Only the tests, the smoke check and
 * the bench's CPU-baseline leg use this file; the CUDA library never links it.
 *
 * The recurrence (Gated DeltaNet, as summarised in the onedev.kr write-up of
 * the FlashQLA AICon 2026 talk, paragraph on the linear-attention background:
 * "the state is accumulated in a d x d matrix"; paragraph on the effective
 * sliding window: "alpha in (0,1), K L2-normalised"):
 *
 *     S_t = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *     o_t = S_t q_t,        alpha_t = exp(g_t),
 *
 * with S_t a d_v x d_k matrix (row index = value dim, column index = key dim).
 * Evaluated literally as: S <- alpha S;  S <- S + beta (v - S k) k^T;  o = S q.
 *
 * Options: q and k may be L2-normalised per token (x / sqrt(sum x^2 + 1e-6))
 * and q is multiplied by `scale` after normalisation.
 *
 * Backward: reverse-mode differentiation of the same token loop (back-
 * propagation through time), with the forward states re-computed from
 * checkpoints taken every CKPT tokens.
 *
 * Layout: tokens packed [T_total, H, D] row-major, sequences given by the
 * int64 offsets cu[0..N] (cu[0] = 0, cu[N] = T_total); states [N, H, Dv, Dk].
 * All arrays are double.  Pairs (sequence, head) are independent and are
 * distributed over OpenMP threads.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define CKPT 64
#define L2EPS 1e-6

/* y = (normalise ? x / sqrt(|x|^2 + eps) : x) * mul; returns the norm used. */
static double prep(const double *x, int d, int normalise, double mul, double *y) {
    double n = 1.0;
    if (normalise) {
        double s = 0.0;
        for (int i = 0; i < d; ++i) s += x[i] * x[i];
        n = sqrt(s + L2EPS);
    }
    for (int i = 0; i < d; ++i) y[i] = x[i] / n * mul;
    return n;
}

/* One token of the recurrence applied to S (Dv x Dk) in place. */
static void step(double *S, int Dk, int Dv, double alpha, double beta,
                 const double *kh, const double *v, double *tmp /* Dv */) {
    for (int a = 0; a < Dv; ++a)
        for (int b = 0; b < Dk; ++b) S[a * Dk + b] *= alpha;
    for (int a = 0; a < Dv; ++a) {
        double sk = 0.0;
        for (int b = 0; b < Dk; ++b) sk += S[a * Dk + b] * kh[b];
        tmp[a] = beta * (v[a] - sk);
    }
    for (int a = 0; a < Dv; ++a)
        for (int b = 0; b < Dk; ++b) S[a * Dk + b] += tmp[a] * kh[b];
}

int gdn_oracle_fwd(long T_total, int H, int Dk, int Dv, int N, const long *cu,
                   const double *q, const double *k, const double *v,
                   const double *g, const double *beta, const double *S0,
                   int l2norm, double scale, double *o, double *ST, int nthreads) {
    (void)T_total;
    if (nthreads <= 0) nthreads = 1;
    long npair = (long)N * H;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (long p = 0; p < npair; ++p) {
        int n = (int)(p / H), h = (int)(p % H);
        double *S = (double *)malloc(sizeof(double) * Dv * Dk);
        double *qh = (double *)malloc(sizeof(double) * Dk);
        double *kh = (double *)malloc(sizeof(double) * Dk);
        double *tmp = (double *)malloc(sizeof(double) * Dv);
        if (S0) memcpy(S, S0 + p * Dv * Dk, sizeof(double) * Dv * Dk);
        else memset(S, 0, sizeof(double) * Dv * Dk);
        for (long t = cu[n]; t < cu[n + 1]; ++t) {
            long r = t * H + h;
            prep(q + r * Dk, Dk, l2norm, scale, qh);
            prep(k + r * Dk, Dk, l2norm, 1.0, kh);
            step(S, Dk, Dv, exp(g[r]), beta[r], kh, v + r * Dv, tmp);
            for (int a = 0; a < Dv; ++a) {
                double acc = 0.0;
                for (int b = 0; b < Dk; ++b) acc += S[a * Dk + b] * qh[b];
                o[r * Dv + a] = acc;
            }
        }
        if (ST) memcpy(ST + p * Dv * Dk, S, sizeof(double) * Dv * Dk);
        free(S); free(qh); free(kh); free(tmp);
    }
    return 0;
}

/*
 * Backward.  With D = dL/dS_t (including everything that flows back from later
 * tokens) and P = S_{t-1}, u = v - alpha P k:
 *   D    += dO_t q^T                      (o_t = S_t q)
 *   dq    = S_t^T dO_t
 *   dv    = beta D k
 *   dbeta = <D k, u>
 *   dk    = beta D^T u - alpha beta P^T D k
 *   dg    = alpha <D, P (I - beta k k^T)>
 *   D    <- alpha D (I - beta k k^T)      (= dL/dS_{t-1})
 * then the normalisation Jacobians map dq^, dk^ back to the raw q, k.
 */
int gdn_oracle_bwd(long T_total, int H, int Dk, int Dv, int N, const long *cu,
                   const double *q, const double *k, const double *v,
                   const double *g, const double *beta, const double *S0,
                   const double *dO, const double *dST, int l2norm, double scale,
                   double *dq, double *dk, double *dv, double *dg, double *dbeta,
                   double *dS0, int nthreads) {
    (void)T_total;
    if (nthreads <= 0) nthreads = 1;
    long npair = (long)N * H;
    long DD = (long)Dv * Dk;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (long p = 0; p < npair; ++p) {
        int n = (int)(p / H), h = (int)(p % H);
        long t0 = cu[n], t1 = cu[n + 1], L = t1 - t0;
        long nblk = (L + CKPT - 1) / CKPT;
        double *ck = (double *)malloc(sizeof(double) * DD * (nblk > 0 ? nblk : 1));
        double *st = (double *)malloc(sizeof(double) * DD * (CKPT + 1));
        double *S = (double *)malloc(sizeof(double) * DD);
        double *D = (double *)malloc(sizeof(double) * DD);
        double *qh = (double *)malloc(sizeof(double) * Dk);
        double *kh = (double *)malloc(sizeof(double) * Dk);
        double *tmp = (double *)malloc(sizeof(double) * Dv);
        double *Dk_ = (double *)malloc(sizeof(double) * Dv);
        double *Pk = (double *)malloc(sizeof(double) * Dv);
        double *u = (double *)malloc(sizeof(double) * Dv);
        double *dqh = (double *)malloc(sizeof(double) * Dk);
        double *dkh = (double *)malloc(sizeof(double) * Dk);

        /* forward, keeping the state at the start of every block */
        if (S0) memcpy(S, S0 + p * DD, sizeof(double) * DD);
        else memset(S, 0, sizeof(double) * DD);
        for (long t = t0; t < t1; ++t) {
            if ((t - t0) % CKPT == 0) memcpy(ck + ((t - t0) / CKPT) * DD, S, sizeof(double) * DD);
            long r = t * H + h;
            prep(k + r * Dk, Dk, l2norm, 1.0, kh);
            step(S, Dk, Dv, exp(g[r]), beta[r], kh, v + r * Dv, tmp);
        }

        if (dST) memcpy(D, dST + p * DD, sizeof(double) * DD);
        else memset(D, 0, sizeof(double) * DD);

        for (long blk = nblk - 1; blk >= 0; --blk) {
            long b0 = t0 + blk * CKPT;
            long b1 = b0 + CKPT < t1 ? b0 + CKPT : t1;
            /* st[i] = state before token b0+i; st[i+1] = after it */
            memcpy(st, ck + blk * DD, sizeof(double) * DD);
            for (long t = b0; t < b1; ++t) {
                long i = t - b0, r = t * H + h;
                memcpy(st + (i + 1) * DD, st + i * DD, sizeof(double) * DD);
                prep(k + r * Dk, Dk, l2norm, 1.0, kh);
                step(st + (i + 1) * DD, Dk, Dv, exp(g[r]), beta[r], kh, v + r * Dv, tmp);
            }
            for (long t = b1 - 1; t >= b0; --t) {
                long i = t - b0, r = t * H + h;
                const double *P = st + i * DD, *St = st + (i + 1) * DD;
                double nq = prep(q + r * Dk, Dk, l2norm, scale, qh);
                double nk = prep(k + r * Dk, Dk, l2norm, 1.0, kh);
                double al = exp(g[r]), be = beta[r];
                const double *dOt = dO + r * Dv;
                const double *vt = v + r * Dv;
                /* o_t = S_t qh */
                for (int a = 0; a < Dv; ++a)
                    for (int b = 0; b < Dk; ++b) D[a * Dk + b] += dOt[a] * qh[b];
                for (int b = 0; b < Dk; ++b) {
                    double acc = 0.0;
                    for (int a = 0; a < Dv; ++a) acc += St[a * Dk + b] * dOt[a];
                    dqh[b] = acc;
                }
                /* S_t = alpha P - alpha beta P k k^T + beta v k^T */
                for (int a = 0; a < Dv; ++a) {
                    double s1 = 0.0, s2 = 0.0;
                    for (int b = 0; b < Dk; ++b) {
                        s1 += D[a * Dk + b] * kh[b];
                        s2 += P[a * Dk + b] * kh[b];
                    }
                    Dk_[a] = s1;
                    Pk[a] = s2;
                    u[a] = vt[a] - al * s2;
                }
                double dbe = 0.0, dDP = 0.0, dkpk = 0.0;
                for (int a = 0; a < Dv; ++a) {
                    dv[r * Dv + a] = be * Dk_[a];
                    dbe += Dk_[a] * u[a];
                    dkpk += Dk_[a] * Pk[a];
                }
                for (long e = 0; e < DD; ++e) dDP += D[e] * P[e];
                for (int b = 0; b < Dk; ++b) {
                    double s1 = 0.0, s2 = 0.0;
                    for (int a = 0; a < Dv; ++a) {
                        s1 += D[a * Dk + b] * u[a];
                        s2 += P[a * Dk + b] * Dk_[a];
                    }
                    dkh[b] = be * s1 - al * be * s2;
                }
                dbeta[r] = dbe;
                dg[r] = al * (dDP - be * dkpk);
                for (int a = 0; a < Dv; ++a)
                    for (int b = 0; b < Dk; ++b)
                        D[a * Dk + b] = al * (D[a * Dk + b] - be * Dk_[a] * kh[b]);
                /* chain through the (optional) normalisation and the q scale */
                if (l2norm) {
                    double cq = 0.0, ck2 = 0.0;
                    /* qh = scale * q / nq ; kh = k / nk */
                    for (int b = 0; b < Dk; ++b) {
                        cq += (q[r * Dk + b] / nq) * dqh[b];
                        ck2 += (k[r * Dk + b] / nk) * dkh[b];
                    }
                    for (int b = 0; b < Dk; ++b) {
                        dq[r * Dk + b] = scale * (dqh[b] - (q[r * Dk + b] / nq) * cq) / nq;
                        dk[r * Dk + b] = (dkh[b] - (k[r * Dk + b] / nk) * ck2) / nk;
                    }
                } else {
                    for (int b = 0; b < Dk; ++b) {
                        dq[r * Dk + b] = scale * dqh[b];
                        dk[r * Dk + b] = dkh[b];
                    }
                }
            }
        }
        if (dS0) memcpy(dS0 + p * DD, D, sizeof(double) * DD);
        free(ck); free(st); free(S); free(D); free(qh); free(kh); free(tmp);
        free(Dk_); free(Pk); free(u); free(dqh); free(dkh);
    }
    return 0;
}

int gdn_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
