/*
 * gdn_oracle.c -- float64 CPU oracle for the gated delta rule.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or load this
 * file: it exists so that tests, the smoke check and the benchmark's CPU-baseline
 * leg can compare the CUDA library against a plain, slow, obviously correct
 * reference. It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (sources are the three pages the method is taken from):
 *
 *   Forward, per value head h of batch row b, kv head hk = h / (Hv/Hk)
 *   (mlx issue #4614 "mx.fast.gated_delta_update VJP: wrong gradient w.r.t. g",
 *    the "Recurrence used for the references" statement and the repro script's
 *    `recurrence()`; S is [Dv, Dk], S_0 = 0 unless given):
 *
 *       S <- g_t * S                      (decay first)
 *       u  = S k_t                        (prediction from the decayed state)
 *       delta = beta_t * (v_t - u)
 *       S <- S + outer(delta, k_t)        (rank-1 delta-rule write)
 *       y_t = S q_t                       (readout of the post-update state)
 *
 *   plus chunk checkpoints ckpt[c] = the state before step c*C (mlx-lm PR #1217
 *   "Add Metal VJP kernel for gated_delta_update", section "What this PR adds":
 *   checkpoints on fixed-size chunks, forward-with-save then a reverse sweep).
 *
 *   Backward: the exact vector-Jacobian product of that forward with respect to
 *   q, k, v, g, beta and S_0, for cotangents dy (and dS_T on the final state).
 *   The pages print no backward formula; it is the chain rule applied, in reverse
 *   time, to the five lines above (written out in oracle_bwd below). dq and dk of
 *   a kv head are the sums over the value heads that read it, added in ascending
 *   value-head order.
 *
 * Parity status: every function here is pinned by tests that do not use this
 * file's arithmetic (central finite differences, an independent forward-mode
 * tangent propagation, torch float64 autograd of the unrolled loop, closed forms
 * for g=0 / g=1,beta=0 / T=1 / orthonormal keys / a fixed unit key, invariants).
 *
 * Memory: the backward keeps one state per chunk boundary and re-runs each chunk
 * from its checkpoint to get the states inside it. Re-running the same float64
 * operations on the same stored state reproduces the same values bit for bit, so
 * this changes memory use only, not the result.
 *
 * Gates (oracle_gates_fwd / oracle_gates_bwd): the decay and write strength computed
 *   from the layer's trainable gate inputs. mlx-lm PR #1217 ("Correctness") checks the
 *   gradients of eight trainable inputs, q, k, v, a, b, A_log, dt_bias and the state,
 *   but no page prints how g and beta follow from a, b, A_log and dt_bias. The reading
 *   taken is the public mlx-lm Qwen3-Next / Qwen3.5 linear-attention layer's:
 *       log g[b,t,h] = -exp(A_log[h]) * softplus(a[b,t,h] + dt_bias[h]),  g = exp(log g)
 *       beta[b,t,h]  = sigmoid(b[b,t,h])
 *   and its VJP goes through log g (mlx issue #4614 warns that the g-gradient is what a
 *   log_g parameterisation trains through): d(log g) = g * dg, never dg / something.
 *
 * Build: plain C99, no fused multiply-add contraction (-ffp-contract=off), optional
 * OpenMP over independent (batch row, value head) pairs.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int B, T, Hk, Hv, Dk, Dv; /* sizes */
    int C;                    /* chunk size of the checkpoints (> 0) */
} oracle_shape;

enum { ORACLE_OK = 0, ORACLE_EINVAL = -1, ORACLE_ENOMEM = -2 };

/* Row-major offsets of the layouts shared with the library under test:
 * q, k [B, T, Hk, Dk]; v, y, dy [B, T, Hv, Dv]; g, beta [B, T, Hv];
 * states [B, Hv, Dv, Dk]; ckpt [B, Hv, NC, Dv, Dk]. */
static size_t off_qk(const oracle_shape *s, int b, int t, int hk) {
    return (((size_t)b * s->T + t) * s->Hk + hk) * (size_t)s->Dk;
}
static size_t off_v(const oracle_shape *s, int b, int t, int h) {
    return (((size_t)b * s->T + t) * s->Hv + h) * (size_t)s->Dv;
}
/* per-value-head rows of dq/dk before the kv-head sum: [B, T, Hv, Dk] */
static size_t off_qh(const oracle_shape *s, int b, int t, int h) {
    return (((size_t)b * s->T + t) * s->Hv + h) * (size_t)s->Dk;
}
static size_t off_gate(const oracle_shape *s, int b, int t, int h) {
    return ((size_t)b * s->T + t) * s->Hv + h;
}
static size_t off_state(const oracle_shape *s, int b, int h) {
    return ((size_t)b * s->Hv + h) * (size_t)s->Dv * s->Dk;
}
static int n_chunks(const oracle_shape *s) { return (s->T + s->C - 1) / s->C; }

static int shape_ok(const oracle_shape *s) {
    return s && s->B > 0 && s->T > 0 && s->Hk > 0 && s->Hv > 0 && s->Dk > 0 && s->Dv > 0 &&
           s->C > 0 && s->Hv % s->Hk == 0;
}

int oracle_n_chunks(const oracle_shape *s) { return shape_ok(s) ? n_chunks(s) : -1; }

/* One forward step on state S [Dv, Dk], in the order the recurrence states it.
 * Writes u (the prediction) and delta; y_t if yt != NULL. */
static void step_forward(int Dv, int Dk, double *S, const double *kt, const double *qt,
                         const double *vt, double gt, double bt, double *u, double *delta,
                         double *yt) {
    for (int i = 0; i < Dv; ++i)
        for (int j = 0; j < Dk; ++j) S[(size_t)i * Dk + j] *= gt;          /* S <- g S */
    for (int i = 0; i < Dv; ++i) {
        double acc = 0.0;
        for (int j = 0; j < Dk; ++j) acc += S[(size_t)i * Dk + j] * kt[j];  /* u = S k */
        u[i] = acc;
    }
    for (int i = 0; i < Dv; ++i) delta[i] = bt * (vt[i] - u[i]);            /* delta */
    for (int i = 0; i < Dv; ++i)
        for (int j = 0; j < Dk; ++j) S[(size_t)i * Dk + j] += delta[i] * kt[j]; /* S += delta k^T */
    if (yt)
        for (int i = 0; i < Dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < Dk; ++j) acc += S[(size_t)i * Dk + j] * qt[j];  /* y = S q */
            yt[i] = acc;
        }
}

/* Forward of one value head (b, h). S enters as S_0 and leaves as S_T. Optional
 * outputs: y (the full [B,T,Hv,Dv] tensor, this head's entries written) and
 * ck (this head's NC checkpoints, [NC, Dv, Dk]). */
static void head_forward(const oracle_shape *s, int b, int h, const double *q, const double *k,
                         const double *v, const double *g, const double *beta, double *S,
                         double *y, double *ck, double *u, double *delta) {
    const int rep = s->Hv / s->Hk, hk = h / rep;
    const size_t nstate = (size_t)s->Dv * s->Dk;
    for (int t = 0; t < s->T; ++t) {
        if (ck && t % s->C == 0) memcpy(ck + (size_t)(t / s->C) * nstate, S, nstate * sizeof(double));
        step_forward(s->Dv, s->Dk, S, k + off_qk(s, b, t, hk), q + off_qk(s, b, t, hk),
                     v + off_v(s, b, t, h), g[off_gate(s, b, t, h)], beta[off_gate(s, b, t, h)],
                     u, delta, y ? y + off_v(s, b, t, h) : NULL);
    }
}

/* Forward over all heads. S0 may be NULL (zeros); S_T and ckpt may be NULL (skipped).
 * nthreads <= 0 uses the OpenMP default. */
int oracle_fwd(const oracle_shape *s, const double *q, const double *k, const double *v,
               const double *g, const double *beta, const double *S0, double *y, double *S_T,
               double *ckpt, int nthreads) {
    if (!shape_ok(s) || !q || !k || !v || !g || !beta || !y) return ORACLE_EINVAL;
    const int nheads = s->B * s->Hv;
    const size_t nstate = (size_t)s->Dv * s->Dk;
    int err = ORACLE_OK;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int bh = 0; bh < nheads; ++bh) {
        const int b = bh / s->Hv, h = bh % s->Hv;
        double *S = malloc(nstate * sizeof(double));
        double *u = malloc((size_t)s->Dv * sizeof(double));
        double *delta = malloc((size_t)s->Dv * sizeof(double));
        if (!S || !u || !delta) {
            err = ORACLE_ENOMEM;
        } else {
            if (S0) memcpy(S, S0 + off_state(s, b, h), nstate * sizeof(double));
            else memset(S, 0, nstate * sizeof(double));
            double *ck = ckpt ? ckpt + off_state(s, b, h) * (size_t)n_chunks(s) : NULL;
            head_forward(s, b, h, q, k, v, g, beta, S, y, ck, u, delta);
            if (S_T) memcpy(S_T + off_state(s, b, h), S, nstate * sizeof(double));
        }
        free(S); free(u); free(delta);
    }
    (void)nthreads;
    return err;
}

/* Reverse-time VJP of one value head (b, h). dqh and dkh ([B, T, Hv, Dk], zeroed by
 * the caller) receive this head's own dq and dk; dv, dg, dbeta are written; dS0 (if not
 * NULL) is written.
 *
 * Per step t, going backwards, with Sh = dL/dS_t accumulated so far:
 *   y_t = S_t q_t            ->  Sh += dy_t q_t^T ;       dq_t += S_t^T dy_t
 *   S_t = A + delta k_t^T    ->  ddelta = Sh k_t ;        dk_t += Sh^T delta ;  dA = Sh
 *   delta = beta (v_t - u)   ->  dv_t = beta ddelta ;     dbeta_t = ddelta . (v_t - u) ;
 *                                du = -beta ddelta
 *   u = A k_t                ->  dA += du k_t^T ;         dk_t += A^T du
 *   A = g_t S_{t-1}          ->  dg_t = <dA, S_{t-1}> ;   Sh <- g_t dA   (= dL/dS_{t-1})
 * and dS_0 is Sh after step 0. */
static int head_backward(const oracle_shape *s, int b, int h, const double *q, const double *k,
                         const double *v, const double *g, const double *beta, const double *S0,
                         const double *dy, const double *dS_T, double *dqh, double *dkh,
                         double *dv, double *dg, double *dbeta, double *dS0) {
    const int rep = s->Hv / s->Hk, hk = h / rep, Dv = s->Dv, Dk = s->Dk, C = s->C;
    const int NC = n_chunks(s);
    const size_t nstate = (size_t)Dv * Dk;
    double *ck = malloc((size_t)NC * nstate * sizeof(double));       /* chunk checkpoints */
    double *st = malloc((size_t)(C + 1) * nstate * sizeof(double));  /* states inside a chunk */
    double *us = malloc((size_t)C * Dv * sizeof(double));            /* u per step of the chunk */
    double *ds = malloc((size_t)C * Dv * sizeof(double));            /* delta per step of the chunk */
    double *Sh = malloc(nstate * sizeof(double));
    double *dA = malloc(nstate * sizeof(double));
    double *dd = malloc((size_t)Dv * sizeof(double));
    double *du = malloc((size_t)Dv * sizeof(double));
    int err = ORACLE_OK;
    if (!ck || !st || !us || !ds || !Sh || !dA || !dd || !du) { err = ORACLE_ENOMEM; goto done; }

    /* forward once, keeping only the chunk checkpoints */
    if (S0) memcpy(st, S0 + off_state(s, b, h), nstate * sizeof(double));
    else memset(st, 0, nstate * sizeof(double));
    head_forward(s, b, h, q, k, v, g, beta, st, NULL, ck, us, ds);

    if (dS_T) memcpy(Sh, dS_T + off_state(s, b, h), nstate * sizeof(double));
    else memset(Sh, 0, nstate * sizeof(double));

    for (int c = NC - 1; c >= 0; --c) {
        const int t0 = c * C, len = (t0 + C <= s->T) ? C : s->T - t0;
        /* states S_{t0-1+tau} for tau = 0..len (st[0] is the checkpoint) */
        memcpy(st, ck + (size_t)c * nstate, nstate * sizeof(double));
        for (int tau = 0; tau < len; ++tau) {
            const int t = t0 + tau;
            memcpy(st + (size_t)(tau + 1) * nstate, st + (size_t)tau * nstate, nstate * sizeof(double));
            step_forward(Dv, Dk, st + (size_t)(tau + 1) * nstate, k + off_qk(s, b, t, hk), NULL,
                         v + off_v(s, b, t, h), g[off_gate(s, b, t, h)], beta[off_gate(s, b, t, h)],
                         us + (size_t)tau * Dv, ds + (size_t)tau * Dv, NULL);
        }
        for (int tau = len - 1; tau >= 0; --tau) {
            const int t = t0 + tau;
            const double *Sprev = st + (size_t)tau * nstate;      /* S_{t-1} */
            const double *Scur = st + (size_t)(tau + 1) * nstate; /* S_t */
            const double *qt = q + off_qk(s, b, t, hk), *kt = k + off_qk(s, b, t, hk);
            const double *vt = v + off_v(s, b, t, h), *dyt = dy + off_v(s, b, t, h);
            const double *u = us + (size_t)tau * Dv, *delta = ds + (size_t)tau * Dv;
            const double gt = g[off_gate(s, b, t, h)], bt = beta[off_gate(s, b, t, h)];
            double *dqt = dqh + off_qh(s, b, t, h), *dkt = dkh + off_qh(s, b, t, h);

            /* y_t = S_t q_t */
            for (int i = 0; i < Dv; ++i)
                for (int j = 0; j < Dk; ++j) Sh[(size_t)i * Dk + j] += dyt[i] * qt[j];
            for (int j = 0; j < Dk; ++j) {
                double acc = 0.0;
                for (int i = 0; i < Dv; ++i) acc += Scur[(size_t)i * Dk + j] * dyt[i];
                dqt[j] += acc;
            }
            /* S_t = A + delta k_t^T */
            for (int i = 0; i < Dv; ++i) {
                double acc = 0.0;
                for (int j = 0; j < Dk; ++j) acc += Sh[(size_t)i * Dk + j] * kt[j];
                dd[i] = acc;
            }
            for (int j = 0; j < Dk; ++j) {
                double acc = 0.0;
                for (int i = 0; i < Dv; ++i) acc += Sh[(size_t)i * Dk + j] * delta[i];
                dkt[j] += acc;
            }
            /* delta = beta (v_t - u) */
            double db = 0.0;
            for (int i = 0; i < Dv; ++i) {
                dv[off_v(s, b, t, h) + i] = bt * dd[i];
                db += dd[i] * (vt[i] - u[i]);
                du[i] = -bt * dd[i];
            }
            dbeta[off_gate(s, b, t, h)] = db;
            /* u = A k_t, A = g_t S_{t-1} */
            for (int i = 0; i < Dv; ++i)
                for (int j = 0; j < Dk; ++j)
                    dA[(size_t)i * Dk + j] = Sh[(size_t)i * Dk + j] + du[i] * kt[j];
            for (int j = 0; j < Dk; ++j) {
                double acc = 0.0;
                for (int i = 0; i < Dv; ++i) acc += (gt * Sprev[(size_t)i * Dk + j]) * du[i];
                dkt[j] += acc;
            }
            double dgt = 0.0;
            for (size_t e = 0; e < nstate; ++e) dgt += dA[e] * Sprev[e];
            dg[off_gate(s, b, t, h)] = dgt;
            for (size_t e = 0; e < nstate; ++e) Sh[e] = gt * dA[e];
        }
    }
    if (dS0) memcpy(dS0 + off_state(s, b, h), Sh, nstate * sizeof(double));
done:
    free(ck); free(st); free(us); free(ds); free(Sh); free(dA); free(dd); free(du);
    return err;
}

/* Backward over all heads. S0 and dS_T may be NULL (zeros); dS0 may be NULL (skipped).
 * Heads run in parallel, each into its own dq/dk rows; then dq and dk of every kv head
 * are the sums of its value heads' rows taken in ascending value-head order.
 * nthreads <= 0 uses the OpenMP default. */
int oracle_bwd(const oracle_shape *s, const double *q, const double *k, const double *v,
               const double *g, const double *beta, const double *S0, const double *dy,
               const double *dS_T, double *dq, double *dk, double *dv, double *dg,
               double *dbeta, double *dS0, int nthreads) {
    if (!shape_ok(s) || !q || !k || !v || !g || !beta || !dy || !dq || !dk || !dv || !dg ||
        !dbeta)
        return ORACLE_EINVAL;
    const int rep = s->Hv / s->Hk, nheads = s->B * s->Hv;
    const size_t nh = (size_t)s->B * s->T * s->Hv * s->Dk;
    double *dqh = calloc(nh, sizeof(double));
    double *dkh = calloc(nh, sizeof(double));
    if (!dqh || !dkh) { free(dqh); free(dkh); return ORACLE_ENOMEM; }
    int err = ORACLE_OK;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int bh = 0; bh < nheads; ++bh) {
        const int b = bh / s->Hv, h = bh % s->Hv;
        int e = head_backward(s, b, h, q, k, v, g, beta, S0, dy, dS_T, dqh, dkh, dv, dg, dbeta, dS0);
        if (e) err = e;
    }
    for (int b = 0; b < s->B; ++b)
        for (int t = 0; t < s->T; ++t)
            for (int hk = 0; hk < s->Hk; ++hk) {
                double *dqt = dq + off_qk(s, b, t, hk), *dkt = dk + off_qk(s, b, t, hk);
                for (int j = 0; j < s->Dk; ++j) { dqt[j] = 0.0; dkt[j] = 0.0; }
                for (int h = hk * rep; h < (hk + 1) * rep; ++h) {
                    const double *qh = dqh + off_qh(s, b, t, h), *kh = dkh + off_qh(s, b, t, h);
                    for (int j = 0; j < s->Dk; ++j) { dqt[j] += qh[j]; dkt[j] += kh[j]; }
                }
            }
    free(dqh); free(dkh);
    (void)nthreads;
    return err;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------------------ */
/* Gates. a, b, g, beta, da, db, dg, dbeta are [BT, Hv] (BT = B*T rows); A_log, dt_bias,  */
/* dA_log, ddt_bias are [Hv]. The parameter gradients are sums over the BT rows, added in */
/* ascending row order.                                                                   */

static double softplus_d(double x) { return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x)); }

static double sigmoid_d(double x) {
    if (x >= 0.0) return 1.0 / (1.0 + exp(-x));
    const double e = exp(x);
    return e / (1.0 + e);
}

int oracle_gates_fwd(int BT, int Hv, const double *a, const double *b, const double *A_log,
                     const double *dt_bias, double *g, double *beta) {
    if (BT <= 0 || Hv <= 0 || !a || !b || !A_log || !dt_bias || !g || !beta) return ORACLE_EINVAL;
    for (int i = 0; i < BT; ++i)
        for (int h = 0; h < Hv; ++h) {
            const size_t o = (size_t)i * Hv + h;
            const double log_g = -exp(A_log[h]) * softplus_d(a[o] + dt_bias[h]);
            g[o] = exp(log_g);
            beta[o] = sigmoid_d(b[o]);
        }
    return ORACLE_OK;
}

int oracle_gates_bwd(int BT, int Hv, const double *a, const double *b, const double *A_log,
                     const double *dt_bias, const double *dg, const double *dbeta, double *da,
                     double *db, double *dA_log, double *ddt_bias) {
    if (BT <= 0 || Hv <= 0 || !a || !b || !A_log || !dt_bias || !dg || !dbeta || !da || !db ||
        !dA_log || !ddt_bias)
        return ORACLE_EINVAL;
    for (int h = 0; h < Hv; ++h) { dA_log[h] = 0.0; ddt_bias[h] = 0.0; }
    for (int i = 0; i < BT; ++i)
        for (int h = 0; h < Hv; ++h) {
            const size_t o = (size_t)i * Hv + h;
            const double A = exp(A_log[h]);
            const double x = a[o] + dt_bias[h];
            const double log_g = -A * softplus_d(x);
            const double dlog_g = exp(log_g) * dg[o];        /* d(log g) = g dg */
            const double dx = dlog_g * (-A) * sigmoid_d(x);   /* softplus' = sigmoid */
            da[o] = dx;
            ddt_bias[h] += dx;
            dA_log[h] += dlog_g * log_g;                      /* d(log g)/d(A_log) = log g */
            const double bt = sigmoid_d(b[o]);
            db[o] = dbeta[o] * bt * (1.0 - bt);
        }
    return ORACLE_OK;
}
