/*
 * TEST INFRASTRUCTURE ONLY - fp64 CPU oracle for causal kernel (linear)
 * attention with a per-head scalar decay (RetNet retention).
 *
 * Only tests/, __graft_entry__.smoke() and bench.py (its cpu_baseline leg
 * and its reference arm) may load this library.  The product path
 * (retnet_retention_gb300) never links, loads or calls it, and this file
 * shares no code, header or table with the CUDA kernels.
 *
 * What it computes is the plain definition, the recurrent form, one token
 * at a time, in fp64, on fp64 copies of the exact input values:
 *
 *   for t = 0 .. T-1:
 *       q~ = phi(q_t),  k~ = phi(k_t)                 phi = elu+1 or identity
 *       S  = gamma * S + k~ v_t^T                      (d_k x d_v)
 *       z  = gamma * z + k~                            (d_k)
 *       o_t = q~^T S          [ / (q~^T z + eps)       if normalising,
 *                               / max(|q~^T z|, 1)    with the floored normaliser ]
 *
 * Sources (web pages on retention / linear attention):
 *  - "Linear attention" (zerotofrontier, Chapter 21 section 21.2), box
 *    "Causal linear attention, recurrent form": S_t = S_{t-1} + phi(k_t) v_t^T,
 *    z_t = z_{t-1} + phi(k_t), o_t = S_t^T phi(q_t) / z_t^T phi(q_t); rows of
 *    S index features, columns index value dimensions; an eps such as 1e-6
 *    is added to the denominator.  The interview box "Causal linear
 *    attention, recurrent and parallel, plus the decode step" fixes that each
 *    token is included in its own sum (update first, then read).
 *  - "RetNet" (bembew), section "Recurrent Representation":
 *    S_n = gamma S_{n-1} + K_n^T V_n, O_n = Q_n S_n, S of shape d_k x d_v.
 *  - "Efficient and Sparse Transformers" (temporalbook section 12.5),
 *    subsection 3: phi(x) = elu(x) + 1; subsection 6 "Linear Attention as a
 *    Special Case": linear attention is retention with gamma = 1.
 *  - "Linear Attention, RWKV, and RetNet" (temporalbook section 13.3),
 *    subsection 4: the generic "decay the old state, add, read out" loop.
 *  - Non-causal form: "Linear attention" (zerotofrontier 21.2), box "Linear
 *    attention": O = diag(phi(Q)(phi(K)^T 1))^-1 phi(Q)(phi(K)^T V).
 *  - Floored normaliser: same page, section "Its normalizer is unstable" and
 *    the box "An LSTM whose cell is linear attention": the matrix LSTM divides
 *    C_t q_t by max(|n_t^T q_t|, 1), n_t the normaliser decayed with the state's
 *    gate; RetNet divides each row of its scores by the absolute value of the
 *    row's sum, clamped below at 1 (the same number: that row sum is q^T z).
 *  - Per-token decay (oracle_recurrent_gated): "Linear Attention, RWKV, and
 *    RetNet" (temporalbook section 13.3), subsection 4 "The Unifying Picture":
 *    decay the old state by G_t, add k_t^T v_t, read out; in the selective
 *    (input-dependent) case G_t depends on the token.  "Efficient and Sparse
 *    Transformers" (temporalbook section 12.5), "Gated Linear Attention:
 *    Toward Input-Dependent Forgetting": RetNet is G_t = gamma 1.  Here G_t is
 *    a_t 1, one scalar per head and token, given as log a_t.
 *
 * Readings where the pages are silent:
 *  - a per-token gate a_t multiplies the state of the step before (S_{t-1}) at
 *    step t, like gamma, and decays z the same way;
 *  - with gamma < 1 and the normaliser on, z decays with the same gamma as S
 *    (the pages never combine the two; the xLSTM box on the "Linear
 *    attention" page decays its normaliser with the same gate as its state);
 *  - eps is added after the dot product, only when normalising with eps; the
 *    floored normaliser has no eps.
 *
 * Compile-time mutants (ORACLE_MUTANT=n) exist only so that the pin tests can
 * show that each plausible mistake is caught; the default build has none.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* elu(x) + 1: x + 1 for x > 0, e^x otherwise ("Linear attention", box
 * "Linear attention by hand on three tokens"). */
static inline double phi_elu1(double x) { return x > 0.0 ? x + 1.0 : exp(x); }

static void feature(const double* x, double* out, long n, int phi)
{
    for (long i = 0; i < n; ++i) {
#if ORACLE_MUTANT == 6 /* mutant: elu without the +1 */
        out[i] = phi ? (x[i] > 0.0 ? x[i] : exp(x[i]) - 1.0) : x[i];
#else
        out[i] = phi ? phi_elu1(x[i]) : x[i];
#endif
    }
}

/*
 * Causal recurrent form over a batch of independent (b, h) sequences.
 *
 *   Q, K : [B][H][T][dk]     V : [B][H][T][dv]
 *   gamma : [H] (per-head decay), or log_a : [B][H][T] (log of a per-token
 *           decay a_t; exactly one of the two is given)
 *   S0   : [B][H][dk][dv] or NULL (zero state)     z0 : [B][H][dk] or NULL
 *   O    : [B][H][T][dv]     S_out : [B][H][dk][dv] or NULL   z_out : [B][H][dk] or NULL
 *   normalize: 0 none, 1 divide by q~^T z + eps, 2 divide by max(|q~^T z|, 1)
 *
 * Returns 0, or -1 when a scratch allocation fails.
 */
static int recurrent(const double* Q, const double* K, const double* V,
                     const double* gamma, const double* log_a, long B, long H, long T,
                     long dk, long dv, int phi, int normalize, double eps,
                     const double* S0, const double* z0,
                     double* O, double* S_out, double* z_out)
{
    int failed = 0;
    long BH = B * H;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (long bh = 0; bh < BH; ++bh) {
        const long h = bh % H;
        double* S = (double*)malloc(sizeof(double) * (size_t)(dk * dv));
        double* z = (double*)malloc(sizeof(double) * (size_t)dk);
        double* qf = (double*)malloc(sizeof(double) * (size_t)dk);
        double* kf = (double*)malloc(sizeof(double) * (size_t)dk);
        if (!S || !z || !qf || !kf) {
            failed = 1;
            free(S); free(z); free(qf); free(kf);
            continue;
        }
        if (S0) memcpy(S, S0 + bh * dk * dv, sizeof(double) * (size_t)(dk * dv));
        else memset(S, 0, sizeof(double) * (size_t)(dk * dv));
        if (z0) memcpy(z, z0 + bh * dk, sizeof(double) * (size_t)dk);
        else memset(z, 0, sizeof(double) * (size_t)dk);

        for (long t = 0; t < T; ++t) {
            const double* q = Q + (bh * T + t) * dk;
            const double* k = K + (bh * T + t) * dk;
            const double* v = V + (bh * T + t) * dv;
            double* o = O + (bh * T + t) * dv;
#if ORACLE_MUTANT == 9 /* mutant: a per-token gate applied one token late */
            const double g = log_a ? (t > 0 ? exp(log_a[bh * T + t - 1]) : 1.0) : gamma[h];
#else
            const double g = log_a ? exp(log_a[bh * T + t]) : gamma[h];
#endif
            feature(q, qf, dk, phi);
            feature(k, kf, dk, phi);
#if ORACLE_MUTANT == 1 /* mutant: read before write (token left out of its own sum) */
            for (long j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (long i = 0; i < dk; ++i) acc += qf[i] * S[i * dv + j];
                o[j] = acc;
            }
#endif
            /* state update: S = gamma S + k~ v^T ; z = gamma z + k~ */
            for (long i = 0; i < dk; ++i) {
                for (long j = 0; j < dv; ++j) {
#if ORACLE_MUTANT == 2 /* mutant: decay applied to the new term as well */
                    S[i * dv + j] = g * (S[i * dv + j] + kf[i] * v[j]);
#elif ORACLE_MUTANT == 3 /* mutant: decay dropped */
                    S[i * dv + j] = S[i * dv + j] + kf[i] * v[j];
#elif ORACLE_MUTANT == 5 /* mutant: outer product written transposed, v k~^T (shapes agree only when dk == dv) */
                    S[i * dv + j] = g * S[i * dv + j] + v[i % dv] * kf[j % dk];
#else
                    S[i * dv + j] = g * S[i * dv + j] + kf[i] * v[j];
#endif
                }
#if ORACLE_MUTANT == 4 /* mutant: normaliser not decayed */
                z[i] = z[i] + kf[i];
#else
                z[i] = g * z[i] + kf[i];
#endif
            }
#if ORACLE_MUTANT != 1
            /* read-out: o = q~^T S (a d_v row) */
            for (long j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (long i = 0; i < dk; ++i) acc += qf[i] * S[i * dv + j];
                o[j] = acc;
            }
#endif
            if (normalize) {
                double den = 0.0;
#if ORACLE_MUTANT == 7 /* mutant: normaliser summed over the feature axis of k only */
                for (long i = 0; i < dk; ++i) den += z[i];
#else
                for (long i = 0; i < dk; ++i) den += qf[i] * z[i];
#endif
                if (normalize == 2) {
#if ORACLE_MUTANT == 8 /* mutant: floor without the absolute value */
                    den = den > 1.0 ? den : 1.0;
#else
                    den = fabs(den) > 1.0 ? fabs(den) : 1.0;
#endif
                } else {
#if ORACLE_MUTANT != 13 /* mutant 13: eps left out of the denominator */
                    den += eps;
#endif
                }
                for (long j = 0; j < dv; ++j) o[j] /= den;
            }
        }
        if (S_out) memcpy(S_out + bh * dk * dv, S, sizeof(double) * (size_t)(dk * dv));
        if (z_out) memcpy(z_out + bh * dk, z, sizeof(double) * (size_t)dk);
        free(S); free(z); free(qf); free(kf);
    }
    return failed ? -1 : 0;
}

int oracle_recurrent(const double* Q, const double* K, const double* V,
                     const double* gamma, long B, long H, long T, long dk, long dv,
                     int phi, int normalize, double eps,
                     const double* S0, const double* z0,
                     double* O, double* S_out, double* z_out)
{
    return recurrent(Q, K, V, gamma, NULL, B, H, T, dk, dv, phi, normalize, eps, S0, z0, O,
                     S_out, z_out);
}

/* The same with a per-token decay: a_t = exp(log_a[b][h][t]) in place of gamma. */
int oracle_recurrent_gated(const double* Q, const double* K, const double* V,
                           const double* log_a, long B, long H, long T, long dk, long dv,
                           int phi, int normalize, double eps,
                           const double* S0, const double* z0,
                           double* O, double* S_out, double* z_out)
{
    return recurrent(Q, K, V, NULL, log_a, B, H, T, dk, dv, phi, normalize, eps, S0, z0, O,
                     S_out, z_out);
}

/*
 * Gradients of the causal recurrent form (the backward pass), for the loss
 * L = sum_t do_t . o_t + <dS_T, S_T> + <dz_T, z_T>, in two sweeps and without
 * storing the states: "Linear attention" (zerotofrontier 21.2), section
 * "Decoding, training, and what each costs": the gradients are cumulative
 * sums too, forward in time for the queries and backward in time for the keys
 * and values (Katharopoulos et al.).  Written out from the recurrence by the
 * chain rule:
 *
 *   forward sweep (t = 0 .. T-1), with S_t, z_t as in the forward pass:
 *       n_t = q~_t S_t,  u_t = q~_t . z_t,  den_t = u_t + eps or max(|u_t|, 1)
 *       dn_t = do_t / den_t            (do_t without the normaliser)
 *       du_t = -(do_t . n_t) / den_t^2 * dden/du   (dden/du = 1, or sign(u_t)
 *              where |u_t| > 1 and 0 elsewhere for the floor)
 *       dq~_t = S_t dn_t + du_t z_t   (a d_k vector: row i of S_t times dn_t)
 *   backward sweep (t = T-1 .. 0), G = dL/dS_t and Gz = dL/dz_t:
 *       G += q~_t^T dn_t,  Gz += du_t q~_t
 *       dv_t = k~_t^T G (a d_v vector),  dk~_t = G v_t + Gz
 *       G = a_t G,  Gz = a_t Gz      (a_t = gamma, or the per-token decay)
 *   and dS_0 = G, dz_0 = Gz after the sweep (gradients of the initial state).
 *   phi: dq = dq~ * phi'(q), phi'(x) = 1 for x > 0, e^x otherwise.
 *
 *   dO : [B][H][T][dv];  dS_T : [B][H][dk][dv] or NULL;  dz_T : [B][H][dk] or NULL
 *   dQ, dK : [B][H][T][dk];  dV : [B][H][T][dv];  dS0 : [B][H][dk][dv] or NULL;
 *   dz0 : [B][H][dk] or NULL.  gamma / log_a, S0, z0 and the flags as in the
 *   forward pass.  Returns 0, or -1 when a scratch allocation fails.
 */
static double phi_grad(double x) { return x > 0.0 ? 1.0 : exp(x); }

/* Token t's own term of dL/dS_t and dL/dz_t: G += q~_t^T dn_t, Gz += du_t q~_t. */
static void add_query_term(double* G, double* Gz, const double* qf, const double* g_o,
                           double den_t, double du_t, long dk, long dv)
{
    for (long i = 0; i < dk; ++i) {
        for (long j = 0; j < dv; ++j) G[i * dv + j] += qf[i] * g_o[j] / den_t;
        Gz[i] += du_t * qf[i];
    }
}

static int recurrent_bwd(const double* Q, const double* K, const double* V,
                         const double* gamma, const double* log_a, long B, long H, long T,
                         long dk, long dv, int phi, int normalize, double eps,
                         const double* S0, const double* z0, const double* dO,
                         const double* dS_T, const double* dz_T,
                         double* dQ, double* dK, double* dV, double* dS0, double* dz0)
{
    int failed = 0;
    long BH = B * H;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (long bh = 0; bh < BH; ++bh) {
        const long h = bh % H;
        double* S = (double*)malloc(sizeof(double) * (size_t)(dk * dv));
        double* z = (double*)malloc(sizeof(double) * (size_t)dk);
        double* qf = (double*)malloc(sizeof(double) * (size_t)dk);
        double* kf = (double*)malloc(sizeof(double) * (size_t)dk);
        double* n = (double*)malloc(sizeof(double) * (size_t)dv);
        double* den = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
        double* du = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
        if (!S || !z || !qf || !kf || !n || !den || !du) {
            failed = 1;
            free(S); free(z); free(qf); free(kf); free(n); free(den); free(du);
            continue;
        }
        /* ---- forward sweep: the states, the denominators, dq */
        if (S0) memcpy(S, S0 + bh * dk * dv, sizeof(double) * (size_t)(dk * dv));
        else memset(S, 0, sizeof(double) * (size_t)(dk * dv));
        if (z0) memcpy(z, z0 + bh * dk, sizeof(double) * (size_t)dk);
        else memset(z, 0, sizeof(double) * (size_t)dk);
        for (long t = 0; t < T; ++t) {
            const double* q = Q + (bh * T + t) * dk;
            const double* k = K + (bh * T + t) * dk;
            const double* v = V + (bh * T + t) * dv;
            const double* g_o = dO + (bh * T + t) * dv;
            const double g = log_a ? exp(log_a[bh * T + t]) : gamma[h];
            feature(q, qf, dk, phi);
            feature(k, kf, dk, phi);
            for (long i = 0; i < dk; ++i) {
                for (long j = 0; j < dv; ++j) S[i * dv + j] = g * S[i * dv + j] + kf[i] * v[j];
                z[i] = g * z[i] + kf[i];
            }
            double u = 0.0;
            for (long i = 0; i < dk; ++i) u += qf[i] * z[i];
            for (long j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (long i = 0; i < dk; ++i) acc += qf[i] * S[i * dv + j];
                n[j] = acc;
            }
            double d = 1.0, dd_du = 0.0;
            if (normalize == 1) {
                d = u + eps;
                dd_du = 1.0;
            } else if (normalize == 2) {
                d = fabs(u) > 1.0 ? fabs(u) : 1.0;
                dd_du = fabs(u) > 1.0 ? (u > 0.0 ? 1.0 : -1.0) : 0.0;
            }
            double don = 0.0;
            for (long j = 0; j < dv; ++j) don += g_o[j] * n[j];
            den[t] = d;
            du[t] = normalize ? -don / (d * d) * dd_du : 0.0;
            double* gq = dQ + (bh * T + t) * dk;
            for (long i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (long j = 0; j < dv; ++j) acc += S[i * dv + j] * g_o[j];
#if ORACLE_MUTANT == 11 /* mutant: dq without the normaliser's term */
                gq[i] = acc / d;
#else
                gq[i] = acc / d + du[t] * z[i];
#endif
                if (phi) gq[i] *= phi_grad(q[i]);
            }
        }
        /* ---- backward sweep: G = dL/dS_t, Gz = dL/dz_t */
        double* G = S;  /* the forward states are no longer needed */
        double* Gz = z;
        if (dS_T) memcpy(G, dS_T + bh * dk * dv, sizeof(double) * (size_t)(dk * dv));
        else memset(G, 0, sizeof(double) * (size_t)(dk * dv));
        if (dz_T) memcpy(Gz, dz_T + bh * dk, sizeof(double) * (size_t)dk);
        else memset(Gz, 0, sizeof(double) * (size_t)dk);
        for (long t = T - 1; t >= 0; --t) {
            const double* q = Q + (bh * T + t) * dk;
            const double* k = K + (bh * T + t) * dk;
            const double* v = V + (bh * T + t) * dv;
            const double* g_o = dO + (bh * T + t) * dv;
            const double g = log_a ? exp(log_a[bh * T + t]) : gamma[h];
            feature(q, qf, dk, phi);
            feature(k, kf, dk, phi);
#if ORACLE_MUTANT != 15 /* mutant 15: dv and dk read G before the token's own term */
            add_query_term(G, Gz, qf, g_o, den[t], du[t], dk, dv);
#endif
            double* gv = dV + (bh * T + t) * dv;
            for (long j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (long i = 0; i < dk; ++i) acc += kf[i] * G[i * dv + j];
                gv[j] = acc;
            }
            double* gk = dK + (bh * T + t) * dk;
            for (long i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (long j = 0; j < dv; ++j) acc += G[i * dv + j] * v[j];
                gk[i] = acc + Gz[i];
#if ORACLE_MUTANT != 16 /* mutant 16: dk without the chain rule through phi */
                if (phi) gk[i] *= phi_grad(k[i]);
#endif
            }
#if ORACLE_MUTANT == 15
            add_query_term(G, Gz, qf, g_o, den[t], du[t], dk, dv);
#endif
#if ORACLE_MUTANT != 10 /* mutant 10: the reverse sweep forgets the decay */
            for (long i = 0; i < dk; ++i) {
                for (long j = 0; j < dv; ++j) G[i * dv + j] *= g;
                Gz[i] *= g;
            }
#endif
        }
        if (dS0) memcpy(dS0 + bh * dk * dv, G, sizeof(double) * (size_t)(dk * dv));
        if (dz0) memcpy(dz0 + bh * dk, Gz, sizeof(double) * (size_t)dk);
        free(S); free(z); free(qf); free(kf); free(n); free(den); free(du);
    }
    return failed ? -1 : 0;
}

int oracle_recurrent_bwd(const double* Q, const double* K, const double* V,
                         const double* gamma, const double* log_a, long B, long H, long T,
                         long dk, long dv, int phi, int normalize, double eps,
                         const double* S0, const double* z0, const double* dO,
                         const double* dS_T, const double* dz_T,
                         double* dQ, double* dK, double* dV, double* dS0, double* dz0)
{
    return recurrent_bwd(Q, K, V, gamma, log_a, B, H, T, dk, dv, phi, normalize, eps, S0, z0,
                         dO, dS_T, dz_T, dQ, dK, dV, dS0, dz0);
}

/*
 * Non-causal form (gamma = 1 only): one summary shared by every query.
 *   S = sum_t k~_t v_t^T,  z = sum_t k~_t,  o_t = q~_t^T S [ / (q~_t^T z + eps) ]
 *   (or / max(|q~_t^T z|, 1) with normalize == 2)
 * Same layouts as oracle_recurrent; S_out/z_out receive S and z.
 */
int oracle_noncausal(const double* Q, const double* K, const double* V,
                     long B, long H, long T, long dk, long dv,
                     int phi, int normalize, double eps,
                     double* O, double* S_out, double* z_out)
{
    int failed = 0;
    long BH = B * H;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (long bh = 0; bh < BH; ++bh) {
        double* S = (double*)calloc((size_t)(dk * dv), sizeof(double));
        double* z = (double*)calloc((size_t)dk, sizeof(double));
        double* f = (double*)malloc(sizeof(double) * (size_t)dk);
        if (!S || !z || !f) {
            failed = 1;
            free(S); free(z); free(f);
            continue;
        }
#if ORACLE_MUTANT == 14 /* mutant: the summary leaves out the last token */
        for (long t = 0; t < T - 1; ++t) {
#else
        for (long t = 0; t < T; ++t) {
#endif
            const double* k = K + (bh * T + t) * dk;
            const double* v = V + (bh * T + t) * dv;
            feature(k, f, dk, phi);
            for (long i = 0; i < dk; ++i) {
                for (long j = 0; j < dv; ++j) S[i * dv + j] += f[i] * v[j];
                z[i] += f[i];
            }
        }
        for (long t = 0; t < T; ++t) {
            const double* q = Q + (bh * T + t) * dk;
            double* o = O + (bh * T + t) * dv;
            feature(q, f, dk, phi);
            for (long j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (long i = 0; i < dk; ++i) acc += f[i] * S[i * dv + j];
                o[j] = acc;
            }
            if (normalize) {
                double den = 0.0;
                for (long i = 0; i < dk; ++i) den += f[i] * z[i];
                den = normalize == 2 ? (fabs(den) > 1.0 ? fabs(den) : 1.0) : den + eps;
                for (long j = 0; j < dv; ++j) o[j] /= den;
            }
        }
        if (S_out) memcpy(S_out + bh * dk * dv, S, sizeof(double) * (size_t)(dk * dv));
        if (z_out) memcpy(z_out + bh * dk, z, sizeof(double) * (size_t)dk);
        free(S); free(z); free(f);
    }
    return failed ? -1 : 0;
}

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
/*
 * Second-order Taylor features ("Linear attention" page, section "A Taylor
 * feature map", box "Taylor features"): for x in R^d
 *
 *   phi(x) = (1, x_1 .. x_d, vec(x x^T) / sqrt(2))        (1 + d + d^2 entries),
 *
 * the constant first, then the d linear features, then the d^2 entries of the
 * outer product in row-major order, so that phi(q)^T phi(k) = 1 + s + s^2 / 2
 * with s = q^T k (the page's theorem).
 *
 *   X : [n][d]     out : [n][1 + d + d*d]
 */
void oracle_taylor_features(const double* X, long n, long d, double* out)
{
    const long df = 1 + d + d * d;
    const double r = 1.0 / sqrt(2.0);
    for (long t = 0; t < n; ++t) {
        const double* x = X + t * d;
        double* f = out + t * df;
#if ORACLE_MUTANT == 17 /* mutant: the constant feature left out */
        f[0] = 0.0;
#else
        f[0] = 1.0;
#endif
#if ORACLE_MUTANT == 18 /* mutant: the linear features left out */
        for (long i = 0; i < d; ++i) f[1 + i] = 0.0;
#else
        for (long i = 0; i < d; ++i) f[1 + i] = x[i];
#endif
        for (long i = 0; i < d; ++i)
            for (long j = 0; j < d; ++j)
#if ORACLE_MUTANT == 12 /* mutant: the outer product without the 1 / sqrt(2) */
                f[1 + d + i * d + j] = x[i] * x[j];
#else
                f[1 + d + i * d + j] = x[i] * x[j] * r;
#endif
    }
}

/*
 * The feature map's transpose Jacobian: given dF = dL/dphi(x) for every row, the
 * gradient dL/dx of the same map (1, x, vec(x x^T) / sqrt(2)) by the chain rule:
 * x_c appears in the linear feature c and in the outer product's entries (c, j)
 * and (i, c), each x_i x_j / sqrt(2), so
 *
 *   dX_c = dF_(1+c) + (1/sqrt 2) sum_j (dF_(1+d+c*d+j) + dF_(1+d+j*d+c)) x_j.
 *
 *   X : [n][d]     dF : [n][1 + d + d*d]     dX : [n][d]
 */
void oracle_taylor_features_bwd(const double* X, const double* dF, long n, long d, double* dX)
{
    const long df = 1 + d + d * d;
    const double r = 1.0 / sqrt(2.0);
    for (long t = 0; t < n; ++t) {
        const double* x = X + t * d;
        const double* g = dF + t * df;
        for (long c = 0; c < d; ++c) {
            double acc = 0.0;
            for (long j = 0; j < d; ++j)
#if ORACLE_MUTANT == 19 /* mutant: only the row of the outer product */
                acc += g[1 + d + c * d + j] * x[j];
#else
                acc += (g[1 + d + c * d + j] + g[1 + d + j * d + c]) * x[j];
#endif
            dX[t * d + c] = g[1 + c] + r * acc;
        }
    }
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
