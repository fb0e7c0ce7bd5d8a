/*
 * lizard_oracle.c -- plain, slow, fp64 CPU reference of the Lizard hybrid
 * attention operator  Y = Y_gate + alpha * Y_anchor.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle that the CUDA path is
 * checked against.  Only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark load it.  It shares no code, header, table or helper
 * with the CUDA library, and it never touches a GPU.
 *
 * What it computes, and where that is stated:
 *
 *   Gate branch (gated linear attention with a learnable gate).
 *     "Lizard: An Efficient Linearization Framework for Large Language Models"
 *     (gist.science/de), section 2 "Kernkomponenten der Architektur", item 1:
 *     a learnable gate Gamma_i = sigmoid(W_gamma x_i) controls the decay of
 *     the past and gives constant-memory inference through incremental updates
 *     of a hidden state.  The same in gist.science/it section 2 "Architettura
 *     Ibrida" and gist.science/pt section 2A "Arquitetura Hibrida".
 *     The pages print no recurrence.  We use the standard GLA recurrence with
 *     a per-token, per-key-dimension decay, rows of S decayed BEFORE the new
 *     outer product is added, and the readout taken after the update:
 *         gamma_t = sigmoid(g_t)                     (g = gate logits)
 *         S_t     = diag(gamma_t) S_{t-1} + k_t^T v_t     S is d_k x d_v
 *         yg_t    = q_t S_t
 *     No normaliser and no feature map (any feature map acts upstream).
 *
 *   Anchor branch (sliding window + meta-memory sinks).
 *     gist.science/de section 2 item 2 "Anchor Window Attention": a local
 *     sliding window of w tokens combined with m learnable meta-memory tokens
 *     that act as attention sinks and stabilise the distribution without
 *     contributing to the output directly (also gist.science/it "Anchor Window
 *     Attention", gist.science/pt "Atencao de Janela Ancora").
 *     Reading: the window holds the w most recent positions INCLUDING the
 *     current one; the meta keys enter the softmax normaliser with value 0;
 *     no scale is applied inside (inputs are pre-scaled):
 *         a_s = q_t . k_s   for max(t-w+1, first) <= s <= t
 *         c_j = q_t . mu_j  for j < m
 *         ya_t = sum_s e^{a_s} v_s / (sum_s e^{a_s} + sum_j e^{c_j})
 *
 *   Combine.  gist.science/de section 2 item 3 "Hybride Ausgabe" (and
 *   gist.science/pt section 2A, last paragraph):  y_t = yg_t + alpha * ya_t.
 *
 *   Decoding with constant memory (gist.science/de section 2 item 1, last
 *   bullet; section 4 "Effizienz"): the decode step applies the same
 *   recurrence to one token, with the window's keys and values kept in a
 *   ring buffer of w slots (token p lives in slot p mod w).
 *
 * Inputs arrive as the exact stored bits (fp32 or bf16) and are widened to
 * fp64 without rounding.  Every sum is a plain left-to-right loop.  There is
 * no chunking, no blocking and no reordering beyond the definitions above.
 *
 * ORACLE_MUTANT: when this file is compiled with -DORACLE_MUTANT=n (n >= 1)
 * one deliberate mistake is planted (see MUT() uses below).  The test-suite
 * builds those variants to show that its pins catch each mistake.  The normal
 * build defines no mutant.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif
#define MUT(n) (ORACLE_MUTANT == (n))

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

/* Widen one stored element to fp64 exactly (bf16 is the top half of fp32). */
static double ld(int dtype, const void *base, size_t idx)
{
    if (dtype == ORACLE_F32)
        return (double)((const float *)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* log(sigmoid(x)) = -log(1 + e^{-x}); each branch keeps exp's argument <= 0. */
double oracle_log_sigmoid(double x)
{
    if (MUT(1))
        return x >= 0 ? -log1p(exp(-x)) : -x - log1p(exp(x));
    return x >= 0 ? -log1p(exp(-x)) : x - log1p(exp(x));
}

/* ------------------------------------------------------------------------ */
/* One (batch, head) unit of the recurrent form.                             */
/* ------------------------------------------------------------------------ */

typedef struct {
    int dtype;
    const void *q, *k, *v, *g; /* [U][L][dk] (v: [U][L][dv]) for this call's units */
    const void *mu;            /* [H][m][dk] */
    double alpha;
    int H, L, dk, dv, w, m;
    const double *S0;   /* [U][dk][dv] initial state, or NULL for zero      */
    const void *hk;     /* [U][hlen][dk] window history (oldest first)     */
    const void *hv;     /* [U][hlen][dv]                                   */
    int hlen;
    double *y;          /* [U][L][dv]                                      */
    double *yg, *ya;    /* optional per-branch outputs, same shape as y    */
    double *S_out;      /* optional [U][dk][dv] final state                */
    int unit0;          /* global index of this call's first unit (b*H+h)  */
    int u_begin, u_end; /* local unit range handled by one worker           */
} fwd_args;

static void forward_unit(const fwd_args *a, int u)
{
    const int L = a->L, dk = a->dk, dv = a->dv, w = a->w, m = a->m;
    const int h = (a->unit0 + u) % a->H;
    const size_t qo = (size_t)u * L * dk, vo = (size_t)u * L * dv;
    double *S = calloc((size_t)dk * dv, sizeof *S);
    double *qt = malloc(sizeof(double) * dk);
    double *yg = malloc(sizeof(double) * dv);
    double *ya = malloc(sizeof(double) * dv);
    double *sc = malloc(sizeof(double) * ((size_t)w + m + 1));
    if (a->S0 && !MUT(10)) /* (mutant 10 drops the initial state) */
        memcpy(S, a->S0 + (size_t)u * dk * dv, sizeof(double) * dk * dv);

    for (int t = 0; t < L; ++t) {
        for (int i = 0; i < dk; ++i)
            qt[i] = ld(a->dtype, a->q, qo + (size_t)t * dk + i);

        /* Gate branch: S <- diag(gamma_t) S + k_t^T v_t ; yg = q_t S. */
        if (MUT(3)) { /* readout before the update */
            for (int j = 0; j < dv; ++j) {
                double acc = 0;
                for (int i = 0; i < dk; ++i) acc += qt[i] * S[(size_t)i * dv + j];
                yg[j] = acc;
            }
        }
        for (int i = 0; i < dk; ++i) {
            double gam = exp(oracle_log_sigmoid(ld(a->dtype, a->g, qo + (size_t)t * dk + i)));
            double ki = ld(a->dtype, a->k, qo + (size_t)t * dk + i);
            for (int j = 0; j < dv; ++j) {
                double vj = ld(a->dtype, a->v, vo + (size_t)t * dv + j);
                if (MUT(2)) /* decay applied after the new term */
                    S[(size_t)i * dv + j] = gam * (S[(size_t)i * dv + j] + ki * vj);
                else
                    S[(size_t)i * dv + j] = gam * S[(size_t)i * dv + j] + ki * vj;
            }
        }
        if (!MUT(3)) {
            for (int j = 0; j < dv; ++j) {
                double acc = 0;
                for (int i = 0; i < dk; ++i) {
                    if (MUT(4) && dk == dv) /* transposed state */
                        acc += qt[i] * S[(size_t)j * dv + i];
                    else
                        acc += qt[i] * S[(size_t)i * dv + j];
                }
                yg[j] = acc;
            }
        }

        /* Anchor branch.  Positions p index history ++ sequence; the
         * history occupies p in [-hlen, -1].  Window: w positions ending at t. */
        int wlen = MUT(5) ? w + 1 : (MUT(6) ? w - 1 : w);
        int p0 = t - wlen + 1;
        if (p0 < -a->hlen) p0 = -a->hlen;
        int n = 0;
        double M = -INFINITY;
        for (int p = p0; p <= t; ++p, ++n) {
            double s = 0;
            for (int i = 0; i < dk; ++i) {
                double kp = p < 0 ? ld(a->dtype, a->hk, ((size_t)u * a->hlen + (a->hlen + p)) * dk + i)
                                  : ld(a->dtype, a->k, qo + (size_t)p * dk + i);
                s += qt[i] * kp;
            }
            sc[n] = s;
            if (s > M) M = s;
        }
        for (int j = 0; j < m; ++j) {
            double s = 0;
            for (int i = 0; i < dk; ++i)
                s += qt[i] * ld(a->dtype, a->mu, ((size_t)h * m + j) * dk + i);
            sc[n + j] = s;
            if (s > M) M = s;
        }
        double Z = 0;
        for (int c = 0; c < n; ++c) Z += exp(sc[c] - M);
        if (!MUT(7))
            for (int j = 0; j < m; ++j) Z += exp(sc[n + j] - M);
        for (int j = 0; j < dv; ++j) ya[j] = 0;
        for (int c = 0; c < n; ++c) {
            int p = p0 + c;
            double pr = exp(sc[c] - M) / Z;
            for (int j = 0; j < dv; ++j) {
                double vp = p < 0 ? ld(a->dtype, a->hv, ((size_t)u * a->hlen + (a->hlen + p)) * dv + j)
                                  : ld(a->dtype, a->v, vo + (size_t)p * dv + j);
                ya[j] += pr * vp;
            }
        }

        /* Combine. */
        for (int j = 0; j < dv; ++j) {
            double out = MUT(8) ? a->alpha * yg[j] + ya[j] : yg[j] + a->alpha * ya[j];
            a->y[vo + (size_t)t * dv + j] = out;
            if (a->yg) a->yg[vo + (size_t)t * dv + j] = yg[j];
            if (a->ya) a->ya[vo + (size_t)t * dv + j] = ya[j];
        }
    }
    if (a->S_out)
        memcpy(a->S_out + (size_t)u * dk * dv, S, sizeof(double) * dk * dv);
    free(S); free(qt); free(yg); free(ya); free(sc);
}

static void *forward_worker(void *p)
{
    const fwd_args *a = p;
    for (int u = a->u_begin; u < a->u_end; ++u)
        forward_unit(a, u);
    return NULL;
}

/*
 * oracle_forward: the operator over U = n_units consecutive (batch, head)
 * units, each a sequence of L tokens.  Unit u (local) has global index
 * unit0 + u and head (unit0 + u) % H.  Inputs q,k,g are [U][L][dk], v is
 * [U][L][dv], mu is [H][m][dk], all in `dtype`.  S0 (nullable) is the
 * initial state [U][dk][dv] in fp64; hk/hv (nullable when hlen == 0) hold the
 * hlen tokens that precede the sequence, oldest first, for the window.
 * Outputs: y [U][L][dv]; yg/ya (nullable) the two branches; S_out (nullable)
 * the final state.  Work is split over nthreads POSIX threads by unit.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_forward(int dtype, const void *q, const void *k, const void *v,
                   const void *g, const void *mu, double alpha,
                   int n_units, int unit0, int H, int L, int dk, int dv, int w, int m,
                   const double *S0, const void *hk, const void *hv, int hlen,
                   double *y, double *yg, double *ya, double *S_out, int nthreads)
{
    if (n_units < 0 || L < 0 || dk < 1 || dv < 1 || w < 1 || m < 0 || H < 1 || hlen < 0)
        return -1;
    if ((dtype != ORACLE_F32 && dtype != ORACLE_BF16) || (m > 0 && !mu) || (hlen > 0 && (!hk || !hv)))
        return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n_units) nthreads = n_units > 0 ? n_units : 1;
    fwd_args base = {dtype, q, k, v, g, mu, alpha, H, L, dk, dv, w, m, S0, hk, hv, hlen,
                     y, yg, ya, S_out, unit0, 0, 0};
    pthread_t *th = malloc(sizeof(pthread_t) * nthreads);
    fwd_args *args = malloc(sizeof(fwd_args) * nthreads);
    for (int i = 0; i < nthreads; ++i) {
        args[i] = base;
        args[i].u_begin = (int)((long long)n_units * i / nthreads);
        args[i].u_end = (int)((long long)n_units * (i + 1) / nthreads);
        pthread_create(&th[i], NULL, forward_worker, &args[i]);
    }
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th); free(args);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Decode step over a ring-buffer state.                                     */
/* ------------------------------------------------------------------------ */

/*
 * oracle_decode_step: one new token for each of B sequences and H heads.
 * q,k,g are [B][H][dk], v is [B][H][dv] in `dtype`; mu is [H][m][dk].
 * State (updated in place): S [B][H][dk][dv] fp64, ring_k [B][H][w][dk] and
 * ring_v [B][H][w][dv] in `dtype` (token p of a sequence sits in slot p mod w),
 * pos [B] = tokens already consumed.  Output y [B][H][dv].
 *
 * The window at position p = pos[b] is the current token plus the tokens
 * max(0, p-w+1) .. p-1 read back from the ring; afterwards the current k, v
 * are written to slot p mod w and pos[b] becomes p + 1.
 */
int oracle_decode_step(int dtype, const void *q, const void *k, const void *v,
                       const void *g, const void *mu, double alpha,
                       int B, int H, int dk, int dv, int w, int m,
                       double *S, void *ring_k, void *ring_v, int64_t *pos, double *y)
{
    if (B < 0 || H < 1 || dk < 1 || dv < 1 || w < 1 || m < 0) return -1;
    if ((dtype != ORACLE_F32 && dtype != ORACLE_BF16) || (m > 0 && !mu)) return -1;
    const size_t es = dtype == ORACLE_F32 ? 4 : 2;
    double *qt = malloc(sizeof(double) * dk), *yg = malloc(sizeof(double) * dv);
    double *ya = malloc(sizeof(double) * dv), *sc = malloc(sizeof(double) * ((size_t)w + m));
    for (int b = 0; b < B; ++b) {
        const int64_t p = pos[b];
        for (int h = 0; h < H; ++h) {
            const size_t u = (size_t)b * H + h;
            double *Su = S + u * dk * dv;
            for (int i = 0; i < dk; ++i) qt[i] = ld(dtype, q, u * dk + i);
            for (int i = 0; i < dk; ++i) {
                double gam = exp(oracle_log_sigmoid(ld(dtype, g, u * dk + i)));
                double ki = ld(dtype, k, u * dk + i);
                for (int j = 0; j < dv; ++j)
                    Su[(size_t)i * dv + j] = gam * Su[(size_t)i * dv + j] + ki * ld(dtype, v, u * dv + j);
            }
            for (int j = 0; j < dv; ++j) {
                double acc = 0;
                for (int i = 0; i < dk; ++i) acc += qt[i] * Su[(size_t)i * dv + j];
                yg[j] = acc;
            }
            /* Window: history tokens first (oldest first), then the current one. */
            int64_t first = p - w + 1;
            if (first < 0) first = 0;
            int n = 0;
            double M = -INFINITY;
            int64_t last = MUT(11) ? p - 1 : p; /* (mutant 11 drops the current token) */
            for (int64_t tau = first; tau <= last; ++tau, ++n) {
                double s = 0;
                size_t slot = (size_t)((MUT(9) ? tau + 1 : tau) % w);
                for (int i = 0; i < dk; ++i) {
                    double kk = tau < p ? ld(dtype, ring_k, (u * w + slot) * dk + i)
                                        : ld(dtype, k, u * dk + i);
                    s += qt[i] * kk;
                }
                sc[n] = s;
                if (s > M) M = s;
            }
            for (int j = 0; j < m; ++j) {
                double s = 0;
                for (int i = 0; i < dk; ++i) s += qt[i] * ld(dtype, mu, ((size_t)h * m + j) * dk + i);
                sc[n + j] = s;
                if (s > M) M = s;
            }
            double Z = 0;
            for (int c = 0; c < n + m; ++c) Z += exp(sc[c] - M);
            for (int j = 0; j < dv; ++j) ya[j] = 0;
            for (int c = 0; c < n; ++c) {
                int64_t tau = first + c;
                size_t slot = (size_t)((MUT(9) ? tau + 1 : tau) % w);
                double pr = exp(sc[c] - M) / Z;
                for (int j = 0; j < dv; ++j) {
                    double vv = tau < p ? ld(dtype, ring_v, (u * w + slot) * dv + j)
                                        : ld(dtype, v, u * dv + j);
                    ya[j] += pr * vv;
                }
            }
            for (int j = 0; j < dv; ++j) y[u * dv + j] = yg[j] + alpha * ya[j];
            /* Ring update: the current token takes slot p mod w. */
            size_t slot = (size_t)(p % w);
            memcpy((char *)ring_k + (u * w + slot) * dk * es, (const char *)k + u * dk * es, dk * es);
            memcpy((char *)ring_v + (u * w + slot) * dv * es, (const char *)v + u * dv * es, dv * es);
        }
        pos[b] = p + 1;
    }
    free(qt); free(yg); free(ya); free(sc);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Product (parallel) form of the gate branch, for tiny inputs only.         */
/* ------------------------------------------------------------------------ */

/*
 * oracle_gla_product_form: the gate branch written as the unrolled
 * recurrence, one term per (t, s) pair, with the decay between s and t taken
 * as the literal product of the sigmoids in between:
 *     yg_t = sum_{s<=t} sum_i q_{t,i} k_{s,i} (prod_{r=s+1..t} sigmoid(g_{r,i})) v_s
 *          + sum_i q_{t,i} (prod_{r=0..t} sigmoid(g_{r,i})) S0[i,:]
 * O(L^3 dk dv); it shares no step with the recurrent loop above except the
 * element widening.  Inputs as oracle_forward for one unit (U = 1); S0 may be
 * NULL.  Output yg [L][dv].
 */
int oracle_gla_product_form(int dtype, const void *q, const void *k, const void *v,
                            const void *g, int L, int dk, int dv, const double *S0, double *yg)
{
    if (L < 0 || dk < 1 || dv < 1) return -1;
    for (int t = 0; t < L; ++t) {
        for (int j = 0; j < dv; ++j) {
            double acc = 0;
            for (int s = 0; s <= t; ++s) {
                for (int i = 0; i < dk; ++i) {
                    double decay = 1.0;
                    for (int r = s + 1; r <= t; ++r)
                        decay *= 1.0 / (1.0 + exp(-ld(dtype, g, (size_t)r * dk + i)));
                    acc += ld(dtype, q, (size_t)t * dk + i) * ld(dtype, k, (size_t)s * dk + i) *
                           decay * ld(dtype, v, (size_t)s * dv + j);
                }
            }
            if (S0) {
                for (int i = 0; i < dk; ++i) {
                    double decay = 1.0;
                    for (int r = 0; r <= t; ++r)
                        decay *= 1.0 / (1.0 + exp(-ld(dtype, g, (size_t)r * dk + i)));
                    acc += ld(dtype, q, (size_t)t * dk + i) * decay * S0[(size_t)i * dv + j];
                }
            }
            yg[(size_t)t * dv + j] = acc;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Backward pass (reverse mode of the forward above).                        */
/* ------------------------------------------------------------------------ */

/*
 * Gradients of a scalar loss with respect to every input of the operator,
 * given dy = dLoss/dy, for sequences that start from the empty state (no S0,
 * no window history): the training case.  Lizard (gist.science/de section 2)
 * trains the gate (item 1), the meta-memory keys (item 2) and alpha (item 3)
 * along with the inputs; the gradients follow from the forward definitions
 * by the chain rule, step by step in reverse:
 *
 *   Combine   y_t = yg_t + alpha ya_t:
 *             dyg_t = dy_t,  dya_t = alpha dy_t,  dalpha += dy_t . ya_t
 *   Gate      yg_t = q_t S_t,  S_t = diag(gamma_t) S_{t-1} + k_t^T v_t,
 *             walked from t = L-1 down to 0 with G = dLoss/dS_t:
 *               G      += q_t^T dyg_t
 *               dq_t   += dyg_t S_t^T  (dq_t[i] = sum_j dyg_t[j] S_t[i][j])
 *               dk_t   += G v_t^T  (dk_t[i] = sum_j G[i][j] v_t[j])
 *               dv_t   += k_t G    (dv_t[j] = sum_i k_t[i] G[i][j])
 *               dgamma_t[i] = sum_j G[i][j] S_{t-1}[i][j]
 *               G       = diag(gamma_t) G          (now dLoss/dS_{t-1})
 *             dg_t = dgamma_t * sigmoid(g_t) * sigmoid(-g_t).
 *   Anchor    p_s = e^{a_s - M} / Z over the window keys s and the sinks j
 *             (value 0), ya_t = sum_s p_s v_s:
 *               dv_s += p_s dya_t;   dp_s = dya_t . v_s  (sinks: dp_j = 0)
 *               da_s  = p_s (dp_s - sum_s' p_s' dp_s'),  dc_j = p_j (0 - same sum)
 *               dq_t += sum_s da_s k_s + sum_j dc_j mu_j
 *               dk_s += da_s q_t;    dmu_j += dc_j q_t
 *
 * The states S_t are those of the forward loop: the walk keeps S at every
 * CKPT-th token and re-runs the identical update to rebuild the states of
 * one block before walking it backwards (memory O((L/CKPT + CKPT) dk dv)
 * instead of O(L dk dv); every value is the forward's, bit for bit).
 */
#define CKPT 64

typedef struct {
    int dtype;
    const void *q, *k, *v, *g, *mu;
    double alpha;
    int H, L, dk, dv, w, m;
    const double *dy;          /* [U][L][dv] */
    double *dq, *dk_, *dv_, *dg; /* [U][L][dk] (dv_: [U][L][dv]) */
    double *dmu;               /* [U][m][dk] per unit */
    double *dalpha;            /* [U] per unit */
    int unit0, u_begin, u_end;
} bwd_args;

/* S <- diag(gamma_t) S + k_t^T v_t for token t of one unit (as in forward_unit). */
static void gate_step(const bwd_args *a, size_t qo, size_t vo, int t, double *S)
{
    const int dk = a->dk, dv = a->dv;
    for (int i = 0; i < dk; ++i) {
        double gam = exp(oracle_log_sigmoid(ld(a->dtype, a->g, qo + (size_t)t * dk + i)));
        double ki = ld(a->dtype, a->k, qo + (size_t)t * dk + i);
        for (int j = 0; j < dv; ++j)
            S[(size_t)i * dv + j] = gam * S[(size_t)i * dv + j] + ki * ld(a->dtype, a->v, vo + (size_t)t * dv + j);
    }
}

static void backward_unit(const bwd_args *a, int u)
{
    const int L = a->L, dk = a->dk, dv = a->dv, w = a->w, m = a->m;
    const int h = (a->unit0 + u) % a->H;
    const size_t qo = (size_t)u * L * dk, vo = (size_t)u * L * dv;
    const size_t SS = (size_t)dk * dv;
    const int nck = (L + CKPT - 1) / CKPT;
    double *ck = calloc((size_t)(nck > 0 ? nck : 1) * SS, sizeof *ck);  /* S before block c */
    double *blk = malloc(sizeof(double) * (CKPT + 1) * SS);             /* S_{t0-1} .. S_{t0+CKPT-1} */
    double *G = calloc(SS, sizeof *G);
    double *qt = malloc(sizeof(double) * dk), *dyt = malloc(sizeof(double) * dv);
    double *ya = malloc(sizeof(double) * dv), *sc = malloc(sizeof(double) * ((size_t)w + m));
    double *dmu = a->dmu + (size_t)u * m * dk;
    double dalpha = 0;

    for (size_t e = 0; e < (size_t)L * dk; ++e) { a->dq[qo + e] = 0; a->dk_[qo + e] = 0; a->dg[qo + e] = 0; }
    for (size_t e = 0; e < (size_t)L * dv; ++e) a->dv_[vo + e] = 0;
    for (size_t e = 0; e < (size_t)m * dk; ++e) dmu[e] = 0;

    /* Checkpoints: the state before every block of CKPT tokens. */
    {
        double *S = calloc(SS, sizeof *S);
        for (int t = 0; t < L; ++t) {
            if (t % CKPT == 0) memcpy(ck + (size_t)(t / CKPT) * SS, S, sizeof(double) * SS);
            gate_step(a, qo, vo, t, S);
        }
        free(S);
    }

    /* Gate branch, walked backwards block by block. */
    for (int c = nck - 1; c >= 0; --c) {
        const int t0 = c * CKPT, t1 = (t0 + CKPT < L) ? t0 + CKPT : L;
        memcpy(blk, ck + (size_t)c * SS, sizeof(double) * SS);
        for (int t = t0; t < t1; ++t) {
            memcpy(blk + (size_t)(t - t0 + 1) * SS, blk + (size_t)(t - t0) * SS, sizeof(double) * SS);
            gate_step(a, qo, vo, t, blk + (size_t)(t - t0 + 1) * SS);
        }
        for (int t = t1 - 1; t >= t0; --t) {
            const double *St = blk + (size_t)(t - t0 + 1) * SS, *Sp = blk + (size_t)(t - t0) * SS;
            for (int i = 0; i < dk; ++i) qt[i] = ld(a->dtype, a->q, qo + (size_t)t * dk + i);
            for (int j = 0; j < dv; ++j) dyt[j] = a->dy[vo + (size_t)t * dv + j];
            for (int i = 0; i < dk; ++i) {
                double acc = 0;
                for (int j = 0; j < dv; ++j) {
                    G[(size_t)i * dv + j] += qt[i] * dyt[j];
                    acc += dyt[j] * St[(size_t)i * dv + j];
                }
                a->dq[qo + (size_t)t * dk + i] += acc;
            }
            for (int i = 0; i < dk; ++i) {
                double acc_k = 0, acc_g = 0;
                for (int j = 0; j < dv; ++j) {
                    acc_k += G[(size_t)i * dv + j] * ld(a->dtype, a->v, vo + (size_t)t * dv + j);
                    acc_g += G[(size_t)i * dv + j] * Sp[(size_t)i * dv + j];
                }
                a->dk_[qo + (size_t)t * dk + i] += acc_k;
                const double gi = ld(a->dtype, a->g, qo + (size_t)t * dk + i);
                const double sg = exp(oracle_log_sigmoid(gi)), sgn = exp(oracle_log_sigmoid(-gi));
                a->dg[qo + (size_t)t * dk + i] = MUT(13) ? acc_g * sg : acc_g * sg * sgn;
            }
            for (int j = 0; j < dv; ++j) {
                double acc = 0;
                for (int i = 0; i < dk; ++i)
                    acc += ld(a->dtype, a->k, qo + (size_t)t * dk + i) * G[(size_t)i * dv + j];
                a->dv_[vo + (size_t)t * dv + j] += acc;
            }
            if (!MUT(12)) /* (mutant 12 forgets to decay the state gradient) */
                for (int i = 0; i < dk; ++i) {
                    double gam = exp(oracle_log_sigmoid(ld(a->dtype, a->g, qo + (size_t)t * dk + i)));
                    for (int j = 0; j < dv; ++j) G[(size_t)i * dv + j] *= gam;
                }
        }
    }

    /* Anchor branch, token by token (no recurrence). */
    for (int t = 0; t < L; ++t) {
        for (int i = 0; i < dk; ++i) qt[i] = ld(a->dtype, a->q, qo + (size_t)t * dk + i);
        for (int j = 0; j < dv; ++j) dyt[j] = a->dy[vo + (size_t)t * dv + j];
        int p0 = t - w + 1;
        if (p0 < 0) p0 = 0;
        const int n = t - p0 + 1;
        double M = -INFINITY;
        for (int c = 0; c < n; ++c) {
            double s = 0;
            for (int i = 0; i < dk; ++i) s += qt[i] * ld(a->dtype, a->k, qo + (size_t)(p0 + c) * dk + i);
            sc[c] = s;
            if (s > M) M = s;
        }
        for (int j = 0; j < m; ++j) {
            double s = 0;
            for (int i = 0; i < dk; ++i) s += qt[i] * ld(a->dtype, a->mu, ((size_t)h * m + j) * dk + i);
            sc[n + j] = s;
            if (s > M) M = s;
        }
        double Z = 0;
        for (int c = 0; c < n + m; ++c) Z += exp(sc[c] - M);
        for (int j = 0; j < dv; ++j) ya[j] = 0;
        for (int c = 0; c < n; ++c) {
            const double pr = exp(sc[c] - M) / Z;
            for (int j = 0; j < dv; ++j) ya[j] += pr * ld(a->dtype, a->v, vo + (size_t)(p0 + c) * dv + j);
        }
        for (int j = 0; j < dv; ++j) dalpha += dyt[j] * ya[j];
        /* dp_s = dya . v_s with dya = alpha dy_t; psum = sum_s p_s dp_s = dya . ya. */
        double psum = 0;
        for (int j = 0; j < dv; ++j) psum += a->alpha * dyt[j] * ya[j];
        for (int c = 0; c < n; ++c) {
            const int s = p0 + c;
            const double pr = exp(sc[c] - M) / Z;
            double dp = 0;
            for (int j = 0; j < dv; ++j) {
                const double vs = ld(a->dtype, a->v, vo + (size_t)s * dv + j);
                dp += a->alpha * dyt[j] * vs;
                a->dv_[vo + (size_t)s * dv + j] += pr * (MUT(16) ? dyt[j] : a->alpha * dyt[j]);
            }
            const double da = MUT(14) ? pr * dp : pr * (dp - psum);
            for (int i = 0; i < dk; ++i) {
                a->dq[qo + (size_t)t * dk + i] += da * ld(a->dtype, a->k, qo + (size_t)s * dk + i);
                a->dk_[qo + (size_t)s * dk + i] += da * qt[i];
            }
        }
        if (!MUT(15)) /* (mutant 15 drops the sinks' gradient) */
            for (int j = 0; j < m; ++j) {
                const double dc = exp(sc[n + j] - M) / Z * (0.0 - psum);
                for (int i = 0; i < dk; ++i) {
                    a->dq[qo + (size_t)t * dk + i] += dc * ld(a->dtype, a->mu, ((size_t)h * m + j) * dk + i);
                    dmu[(size_t)j * dk + i] += dc * qt[i];
                }
            }
    }
    a->dalpha[u] = dalpha;
    free(ck); free(blk); free(G); free(qt); free(dyt); free(ya); free(sc);
}

static void *backward_worker(void *p)
{
    const bwd_args *a = p;
    for (int u = a->u_begin; u < a->u_end; ++u)
        backward_unit(a, u);
    return NULL;
}

/*
 * oracle_backward: gradients of the operator over U = n_units (batch, head)
 * units that start from the empty state.  Inputs as oracle_forward; dy
 * [U][L][dv] fp64.  Outputs (fp64): dq, dk, dg [U][L][dk], dv [U][L][dv],
 * dmu [U][m][dk] and dalpha [U], the last two per unit (the caller sums
 * dmu over the batch for each head and dalpha over all units).
 * Returns 0, or -1 on a bad argument.
 */
int oracle_backward(int dtype, const void *q, const void *k, const void *v, const void *g,
                    const void *mu, double alpha, int n_units, int unit0, int H, int L,
                    int dk, int dv, int w, int m, const double *dy,
                    double *dq, double *dk_out, double *dv_out, double *dg, double *dmu,
                    double *dalpha, int nthreads)
{
    if (n_units < 0 || L < 0 || dk < 1 || dv < 1 || w < 1 || m < 0 || H < 1) return -1;
    if ((dtype != ORACLE_F32 && dtype != ORACLE_BF16) || (m > 0 && !mu)) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n_units) nthreads = n_units > 0 ? n_units : 1;
    bwd_args base = {dtype, q, k, v, g, mu, alpha, H, L, dk, dv, w, m, dy, dq, dk_out, dv_out, dg,
                     dmu, dalpha, unit0, 0, 0};
    pthread_t *th = malloc(sizeof(pthread_t) * nthreads);
    bwd_args *args = malloc(sizeof(bwd_args) * nthreads);
    for (int i = 0; i < nthreads; ++i) {
        args[i] = base;
        args[i].u_begin = (int)((long long)n_units * i / nthreads);
        args[i].u_end = (int)((long long)n_units * (i + 1) / nthreads);
        pthread_create(&th[i], NULL, backward_worker, &args[i]);
    }
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th); free(args);
    return 0;
}
