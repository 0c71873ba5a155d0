/*
 * gdr_oracle.c -- the fp64 CPU oracle for the gated delta rule with a
 * lower-bounded decay.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  It shares no
 * code, header, table or helper with the CUDA library, and never calls it.
 *
 * What it computes (per head, one token at a time, all arithmetic in fp64):
 *
 *   alpha_t = a_min + (1 - a_min) * sigmoid(g_t)
 *           (or, in the log-domain mode, alpha_t = exp(g_min * sigmoid(g_t)))
 *   S_t     = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *   o_t     = S_t q_t
 *
 * S is the dv x dk associative-memory state.  The pages describe the
 * incremental ("delta") rule only in words: a write that corrects what the
 * state already returns for k_t, combined with a position-dependent decay
 * gate ("How to Think About Trillion-Parameter Sparse Multimodal LLMs",
 * section 2.2, Incremental Linear Attention).  The equations above are the
 * plain reading of that rule with a scalar decay per token and head; the
 * lower-bounded decay is the scaled-sigmoid bound of "Trillion-Parameter MoE
 * Multimodal LLMs: How to Evaluate the New Generation", section 3.1, taken in
 * the linear domain with floor a_min.
 *
 * Memory layouts are those of the library's public boundary: q, k [B,H,T,dk],
 * v [B,H,T,dv], g and beta [B,H,T], state [B,H,dk,dv] holding M = S^T
 * (M[i][j] = S[j][i]).  Inputs arrive as float32 arrays; bf16 inputs are
 * widened exactly by the caller, so the oracle sees the very values a GPU
 * kernel would see.  Nothing here is blocked, fused or reordered: the loop
 * below is the recurrence as written.
 *
 * Parity status: every function here is pinned by the CPU tests (explicit
 * unrolled matrix products, the orthonormal-key write/read invariant, closed
 * forms for beta = 0 and a_min = 1, a hand-worked two-step case, and agreement
 * with an independent chunkwise reformulation).  The backward (gdr_oracle_bwd)
 * is pinned by central finite differences of the forward loss for every input
 * element, by exactness in the inputs the loss is linear in (q, v, the initial
 * state), and by the pure-decay closed form at beta = 0.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* alpha = a_min + (1 - a_min) * sigmoid(g), sigmoid(g) = 1 / (1 + e^{-g}). */
double gdr_oracle_alpha(double g, double a_min)
{
    return a_min + (1.0 - a_min) / (1.0 + exp(-g));
}

/*
 * The pages' own form of the bound, in the log domain: log alpha = g_min *
 * sigmoid(g) with g_min < 0 ("Trillion-Parameter MoE Multimodal LLMs: How to
 * Evaluate the New Generation", section 3.1, with g_min = -5; "What a
 * Trillion-Parameter MoE Model Reveals About the Next Stage of LLM Scaling",
 * section 3.2), so alpha = exp(g_min * sigmoid(g)) lies in (e^{g_min}, 1).
 */
double gdr_oracle_alpha_log(double g, double g_min)
{
    return exp(g_min / (1.0 + exp(-g)));
}

/* decay 0: the linear-domain bound (bound = a_min); decay 1: the log-domain bound
 * (bound = g_min). */
static double decay_alpha(int decay, double g, double bound)
{
    return decay == 1 ? gdr_oracle_alpha_log(g, bound) : gdr_oracle_alpha(g, bound);
}

/*
 * One head.  q, k: [T][dk]; v: [T][dv]; g, beta: [T]; init: [dk][dv] (M
 * layout) or NULL for a zero state; out: [T][dv] or NULL; final_state:
 * [dk][dv] (M layout) or NULL.  S is held as S[j][i], j < dv, i < dk.
 */
static void oracle_head(const float *q, const float *k, const float *v,
                        const float *g, const float *beta, int decay, double a_min,
                        const float *init, double *out, double *final_state,
                        int64_t T, int dk, int dv, double *S, double *u)
{
    for (int j = 0; j < dv; ++j)
        for (int i = 0; i < dk; ++i)
            S[(int64_t)j * dk + i] = init ? (double)init[(int64_t)i * dv + j] : 0.0;

    for (int64_t t = 0; t < T; ++t) {
        const float *kt = k + t * dk;
        const float *qt = q + t * dk;
        const float *vt = v + t * dv;
        const double a = decay_alpha(decay, (double)g[t], a_min);
        const double b = (double)beta[t];

        /* u = S k_t */
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i)
                acc += S[(int64_t)j * dk + i] * (double)kt[i];
            u[j] = acc;
        }
        /* S <- a * (S - b * u k_t^T) + b * v_t k_t^T
         *    = a * S (I - b k_t k_t^T) + b v_t k_t^T                  */
        for (int j = 0; j < dv; ++j) {
            const double uj = u[j];
            const double vj = (double)vt[j];
            for (int i = 0; i < dk; ++i) {
                const double ki = (double)kt[i];
                double *s = &S[(int64_t)j * dk + i];
                *s = a * (*s - b * uj * ki) + b * vj * ki;
            }
        }
        /* o_t = S q_t */
        if (out) {
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i)
                    acc += S[(int64_t)j * dk + i] * (double)qt[i];
                out[t * dv + j] = acc;
            }
        }
    }

    if (final_state)
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j)
                final_state[(int64_t)i * dv + j] = S[(int64_t)j * dk + i];
}

typedef struct {
    const float *q, *k, *v, *g, *beta, *init;
    int decay;
    double a_min;
    double *out, *final_state;
    int B, H, dk, dv;
    int64_t T;
    int64_t next;            /* next (b, h) work item, taken atomically */
} job_t;

static void *worker(void *arg)
{
    job_t *jb = (job_t *)arg;
    const int64_t nbh = (int64_t)jb->B * jb->H;
    double *S = (double *)malloc(sizeof(double) * (size_t)jb->dk * (size_t)jb->dv);
    double *u = (double *)malloc(sizeof(double) * (size_t)jb->dv);
    if (!S || !u) {
        free(S);
        free(u);
        return (void *)1;
    }
    for (;;) {
        const int64_t bh = __atomic_fetch_add(&jb->next, 1, __ATOMIC_RELAXED);
        if (bh >= nbh)
            break;
        const int64_t T = jb->T;
        oracle_head(jb->q + bh * T * jb->dk, jb->k + bh * T * jb->dk,
                    jb->v + bh * T * jb->dv, jb->g + bh * T, jb->beta + bh * T,
                    jb->decay, jb->a_min,
                    jb->init ? jb->init + bh * jb->dk * jb->dv : NULL,
                    jb->out ? jb->out + bh * T * jb->dv : NULL,
                    jb->final_state ? jb->final_state + bh * jb->dk * jb->dv : NULL,
                    T, jb->dk, jb->dv, S, u);
    }
    free(S);
    free(u);
    return NULL;
}

/*
 * Full forward over [B,H,T]: the token loop above for every (b, h), spread
 * over nthreads host threads (one whole head per thread at a time, so the
 * arithmetic of each head is the same whatever the thread count).
 * Returns 0 on success, -1 on bad arguments, -2 if memory ran out.
 */
int gdr_oracle_fwd(const float *q, const float *k, const float *v,
                   const float *g, const float *beta, double a_min,
                   const float *init_state, double *out, double *final_state,
                   int B, int H, int64_t T, int dk, int dv, int nthreads, int decay)
{
    if (!q || !k || !v || !g || !beta || B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0)
        return -1;
    if (nthreads < 1)
        nthreads = 1;
    job_t jb = {q, k, v, g, beta, init_state, decay, a_min, out, final_state,
                B, H, dk, dv, T, 0};
    const int64_t nbh = (int64_t)B * H;
    if (nthreads > nbh)
        nthreads = nbh > 0 ? (int)nbh : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th)
        return -2;
    int rc = 0;
    int started = 0;
    for (int i = 1; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, worker, &jb) != 0)
            break;
        started = i;
    }
    if (worker(&jb) != NULL)
        rc = -2;
    for (int i = 1; i <= started; ++i) {
        void *r = NULL;
        pthread_join(th[i], &r);
        if (r != NULL)
            rc = -2;
    }
    free(th);
    return rc;
}

/* One (sequence, head) of a decode step: the recurrence with T = 1 applied in
 * place to M [dk][dv] (fp64, M layout); S is dv x dk scratch. */
static void oracle_decode_one(const float *qt, const float *kt, const float *vt,
                              double a, double b, double *M, double *out, int dk, int dv,
                              double *S)
{
    for (int j = 0; j < dv; ++j)
        for (int i = 0; i < dk; ++i)
            S[(int64_t)j * dk + i] = M[(int64_t)i * dv + j];
    for (int j = 0; j < dv; ++j) {
        double uj = 0.0;
        for (int i = 0; i < dk; ++i)
            uj += S[(int64_t)j * dk + i] * (double)kt[i];
        const double vj = (double)vt[j];
        for (int i = 0; i < dk; ++i) {
            const double ki = (double)kt[i];
            double *s = &S[(int64_t)j * dk + i];
            *s = a * (*s - b * uj * ki) + b * vj * ki;
        }
        double oj = 0.0;
        for (int i = 0; i < dk; ++i)
            oj += S[(int64_t)j * dk + i] * (double)qt[i];
        out[j] = oj;
    }
    for (int j = 0; j < dv; ++j)
        for (int i = 0; i < dk; ++i)
            M[(int64_t)i * dv + j] = S[(int64_t)j * dk + i];
}

typedef struct {
    const float *q, *k, *v, *g, *beta;
    int decay;
    double a_min;
    double *state, *out;
    int64_t NH;
    int dk, dv;
    int64_t next;
} decode_job_t;

static void *decode_worker(void *arg)
{
    decode_job_t *jb = (decode_job_t *)arg;
    double *S = (double *)malloc(sizeof(double) * (size_t)jb->dk * (size_t)jb->dv);
    if (!S)
        return (void *)1;
    for (;;) {
        const int64_t nh = __atomic_fetch_add(&jb->next, 1, __ATOMIC_RELAXED);
        if (nh >= jb->NH)
            break;
        const double a = decay_alpha(jb->decay, (double)jb->g[nh], jb->a_min);
        oracle_decode_one(jb->q + nh * jb->dk, jb->k + nh * jb->dk, jb->v + nh * jb->dv, a,
                          (double)jb->beta[nh], jb->state + nh * jb->dk * jb->dv,
                          jb->out + nh * jb->dv, jb->dk, jb->dv, S);
    }
    free(S);
    return NULL;
}

/*
 * One decode step for N independent sequences: the same recurrence with
 * T = 1, applied in place to state [N,H,dk,dv] (fp64, M layout).
 * q, k [N,H,dk]; v [N,H,dv]; g, beta [N,H]; out [N,H,dv].  The (n, h) pairs
 * are spread over nthreads host threads; each pair's arithmetic is the same
 * whatever the thread count.
 */
int gdr_oracle_decode(const float *q, const float *k, const float *v,
                      const float *g, const float *beta, double a_min,
                      double *state, double *out, int N, int H, int dk, int dv,
                      int nthreads, int decay)
{
    if (!q || !k || !v || !g || !beta || !state || !out || N < 0 || H < 0 ||
        dk <= 0 || dv <= 0)
        return -1;
    decode_job_t jb = {q, k, v, g, beta, decay, a_min, state, out, (int64_t)N * H, dk, dv, 0};
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > jb.NH)
        nthreads = jb.NH > 0 ? (int)jb.NH : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th)
        return -2;
    int rc = 0, started = 0;
    for (int i = 1; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, decode_worker, &jb) != 0)
            break;
        started = i;
    }
    if (decode_worker(&jb) != NULL)
        rc = -2;
    for (int i = 1; i <= started; ++i) {
        void *r = NULL;
        pthread_join(th[i], &r);
        if (r != NULL)
            rc = -2;
    }
    free(th);
    return rc;
}

/* ------------------------------------------------------------------ backward
 *
 * The gradient of L = sum_t <dout_t, o_t> + <dfinal, M_T> with respect to
 * every input, by reverse-mode differentiation of the token loop above: the
 * forward steps are replayed as written and each step is then undone in
 * reverse order.  With S = S_{t-1}, a = alpha_t, b = beta_t, the forward step
 * is
 *     u = S k_t,   r = v_t - a u,   w = b r,   S_t = a S + w k_t^T,   o_t = S_t q_t
 * (S_t = a S (I - b k k^T) + b v k^T written out), so for G = dL/dS_t:
 *     G      += dout_t q_t^T                      (o_t = S_t q_t)
 *     dq_t    = S_t^T dout_t
 *     dw      = G k_t,   dk_t = G^T w + S^T du,   du = -a b dw
 *     dv_t    = b dw,    dbeta_t = dw . r
 *     dalpha  = <G, S> - b (dw . u),   dg_t = dalpha * dalpha/dg
 *     dL/dS_{t-1} = a G + du k_t^T
 * and the initial state's gradient is dL/dS_0.  The states S_{t-1} are kept at
 * every 64th token and the steps between two of them replayed from there,
 * which changes no value: the replay repeats the forward's arithmetic.
 */
#define ORACLE_BWD_SEG 64

/* d alpha / d g for the two decay forms. */
static double decay_dalpha(int decay, double g, double bound)
{
    const double s = 1.0 / (1.0 + exp(-g));
    if (decay == 1)
        return gdr_oracle_alpha_log(g, bound) * bound * s * (1.0 - s);
    return (1.0 - bound) * s * (1.0 - s);
}

/* One forward step of the loop above on S (dv x dk), in place; u is scratch. */
static void oracle_step(double *S, const float *kt, const float *vt, double a, double b,
                        int dk, int dv, double *u)
{
    for (int j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int i = 0; i < dk; ++i)
            acc += S[(int64_t)j * dk + i] * (double)kt[i];
        u[j] = acc;
    }
    for (int j = 0; j < dv; ++j) {
        const double uj = u[j];
        const double vj = (double)vt[j];
        for (int i = 0; i < dk; ++i) {
            const double ki = (double)kt[i];
            double *s = &S[(int64_t)j * dk + i];
            *s = a * (*s - b * uj * ki) + b * vj * ki;
        }
    }
}

/*
 * Backward of one head.  Inputs as oracle_head plus dout [T][dv] (or NULL =
 * zero) and dfinal [dk][dv] (M layout, or NULL = zero).  Outputs (fp64):
 * gq, gk [T][dk]; gv [T][dv]; gg, gb [T]; ginit [dk][dv] (M layout).
 * Scratch: ck ((T / SEG + 1) states), st (SEG + 1 states), G (one state),
 * vec (4 * max(dk, dv)).  Returns 0.
 */
static int oracle_head_bwd(const float *q, const float *k, const float *v, const float *g,
                           const float *beta, int decay, double bound, const float *init,
                           const float *dout, const float *dfinal, double *gq, double *gk,
                           double *gv, double *gg, double *gb, double *ginit, int64_t T,
                           int dk, int dv, double *ck, double *st, double *G, double *vec)
{
    const int64_t SZ = (int64_t)dk * dv;
    double *u = vec, *w = vec + dv, *dw = vec + 2 * dv, *du = vec + 3 * dv;

    /* forward, keeping S_{t-1} at every SEG-th token */
    double *S = st;
    for (int j = 0; j < dv; ++j)
        for (int i = 0; i < dk; ++i)
            S[(int64_t)j * dk + i] = init ? (double)init[(int64_t)i * dv + j] : 0.0;
    for (int64_t t = 0; t < T; ++t) {
        if (t % ORACLE_BWD_SEG == 0)
            memcpy(ck + (t / ORACLE_BWD_SEG) * SZ, S, sizeof(double) * (size_t)SZ);
        oracle_step(S, k + t * dk, v + t * dv, decay_alpha(decay, (double)g[t], bound),
                    (double)beta[t], dk, dv, u);
    }

    /* G = dL/dS_T */
    for (int j = 0; j < dv; ++j)
        for (int i = 0; i < dk; ++i)
            G[(int64_t)j * dk + i] = dfinal ? (double)dfinal[(int64_t)i * dv + j] : 0.0;

    const int64_t nseg = (T + ORACLE_BWD_SEG - 1) / ORACLE_BWD_SEG;
    for (int64_t sg = nseg - 1; sg >= 0; --sg) {
        const int64_t t0 = sg * ORACLE_BWD_SEG;
        const int64_t t1 = t0 + ORACLE_BWD_SEG < T ? t0 + ORACLE_BWD_SEG : T;
        /* replay: st[m] = S_{t0 + m - 1}, m = 0 .. t1 - t0 */
        memcpy(st, ck + sg * SZ, sizeof(double) * (size_t)SZ);
        for (int64_t t = t0; t < t1; ++t) {
            memcpy(st + (t - t0 + 1) * SZ, st + (t - t0) * SZ, sizeof(double) * (size_t)SZ);
            oracle_step(st + (t - t0 + 1) * SZ, k + t * dk, v + t * dv,
                        decay_alpha(decay, (double)g[t], bound), (double)beta[t], dk, dv, u);
        }
        for (int64_t t = t1 - 1; t >= t0; --t) {
            const double *Sp = st + (t - t0) * SZ;      /* S_{t-1} */
            const double *St = st + (t - t0 + 1) * SZ;  /* S_t */
            const float *kt = k + t * dk, *qt = q + t * dk, *vt = v + t * dv;
            const float *dot = dout ? dout + t * dv : NULL;
            const double a = decay_alpha(decay, (double)g[t], bound);
            const double b = (double)beta[t];
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i)
                    acc += Sp[(int64_t)j * dk + i] * (double)kt[i];
                u[j] = acc;
                w[j] = b * ((double)vt[j] - a * acc);
            }
            /* o_t = S_t q_t */
            for (int i = 0; i < dk; ++i) {
                double acc = 0.0;
                if (dot)
                    for (int j = 0; j < dv; ++j)
                        acc += St[(int64_t)j * dk + i] * (double)dot[j];
                gq[t * dk + i] = acc;
            }
            if (dot)
                for (int j = 0; j < dv; ++j)
                    for (int i = 0; i < dk; ++i)
                        G[(int64_t)j * dk + i] += (double)dot[j] * (double)qt[i];
            /* S_t = a S_{t-1} + w k_t^T */
            double dalpha = 0.0;
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) {
                    acc += G[(int64_t)j * dk + i] * (double)kt[i];
                    dalpha += G[(int64_t)j * dk + i] * Sp[(int64_t)j * dk + i];
                }
                dw[j] = acc;
            }
            /* w = b (v - a u) */
            double dbeta = 0.0;
            for (int j = 0; j < dv; ++j) {
                gv[t * dv + j] = b * dw[j];
                dbeta += dw[j] * ((double)vt[j] - a * u[j]);
                dalpha -= b * dw[j] * u[j];
                du[j] = -a * b * dw[j];
            }
            /* u = S_{t-1} k_t; w k_t^T */
            for (int i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dv; ++j)
                    acc += G[(int64_t)j * dk + i] * w[j] + Sp[(int64_t)j * dk + i] * du[j];
                gk[t * dk + i] = acc;
            }
            gb[t] = dbeta;
            gg[t] = dalpha * decay_dalpha(decay, (double)g[t], bound);
            /* dL/dS_{t-1} = a G + du k_t^T */
            for (int j = 0; j < dv; ++j)
                for (int i = 0; i < dk; ++i)
                    G[(int64_t)j * dk + i] = a * G[(int64_t)j * dk + i] + du[j] * (double)kt[i];
        }
    }
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j)
            ginit[(int64_t)i * dv + j] = G[(int64_t)j * dk + i];
    return 0;
}

typedef struct {
    const float *q, *k, *v, *g, *beta, *init, *dout, *dfinal;
    int decay;
    double bound;
    double *gq, *gk, *gv, *gg, *gb, *ginit;
    int B, H, dk, dv;
    int64_t T;
    int64_t next;
} bwd_job_t;

static void *bwd_worker(void *arg)
{
    bwd_job_t *jb = (bwd_job_t *)arg;
    const int64_t nbh = (int64_t)jb->B * jb->H, T = jb->T;
    const int64_t SZ = (int64_t)jb->dk * jb->dv;
    const int64_t nck = T / ORACLE_BWD_SEG + 1;
    const int mx = jb->dk > jb->dv ? jb->dk : jb->dv;
    double *ck = (double *)malloc(sizeof(double) * (size_t)(nck * SZ));
    double *st = (double *)malloc(sizeof(double) * (size_t)((ORACLE_BWD_SEG + 1) * SZ));
    double *G = (double *)malloc(sizeof(double) * (size_t)SZ);
    double *vec = (double *)malloc(sizeof(double) * (size_t)(4 * mx));
    void *rc = NULL;
    if (!ck || !st || !G || !vec) {
        rc = (void *)1;
        goto done;
    }
    for (;;) {
        const int64_t bh = __atomic_fetch_add(&jb->next, 1, __ATOMIC_RELAXED);
        if (bh >= nbh)
            break;
        oracle_head_bwd(jb->q + bh * T * jb->dk, jb->k + bh * T * jb->dk, jb->v + bh * T * jb->dv,
                        jb->g + bh * T, jb->beta + bh * T, jb->decay, jb->bound,
                        jb->init ? jb->init + bh * SZ : NULL,
                        jb->dout ? jb->dout + bh * T * jb->dv : NULL,
                        jb->dfinal ? jb->dfinal + bh * SZ : NULL,
                        jb->gq + bh * T * jb->dk, jb->gk + bh * T * jb->dk,
                        jb->gv + bh * T * jb->dv, jb->gg + bh * T, jb->gb + bh * T,
                        jb->ginit + bh * SZ, T, jb->dk, jb->dv, ck, st, G, vec);
    }
done:
    free(ck);
    free(st);
    free(G);
    free(vec);
    return rc;
}

/*
 * Backward over [B,H,T]: the gradients of L = sum <d_out, out> + <d_final,
 * final_state> with respect to q, k [B,H,T,dk], v [B,H,T,dv], g, beta [B,H,T]
 * and the initial state [B,H,dk,dv] (M layout), for the forward of
 * gdr_oracle_fwd with the same (bound, decay).  d_out and d_final may be NULL
 * (zero).  Heads are spread over nthreads host threads.  Returns 0 on
 * success, -1 on bad arguments, -2 if memory ran out.
 */
int gdr_oracle_bwd(const float *q, const float *k, const float *v, const float *g,
                   const float *beta, double bound, const float *init_state, const float *d_out,
                   const float *d_final, double *gq, double *gk, double *gv, double *gg,
                   double *gbeta, double *ginit, int B, int H, int64_t T, int dk, int dv,
                   int nthreads, int decay)
{
    if (!q || !k || !v || !g || !beta || !gq || !gk || !gv || !gg || !gbeta || !ginit ||
        B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0)
        return -1;
    bwd_job_t jb = {q, k, v, g, beta, init_state, d_out, d_final, decay, bound,
                    gq, gk, gv, gg, gbeta, ginit, B, H, dk, dv, T, 0};
    const int64_t nbh = (int64_t)B * H;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > nbh)
        nthreads = nbh > 0 ? (int)nbh : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th)
        return -2;
    int rc = 0, started = 0;
    for (int i = 1; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, bwd_worker, &jb) != 0)
            break;
        started = i;
    }
    if (bwd_worker(&jb) != NULL)
        rc = -2;
    for (int i = 1; i <= started; ++i) {
        void *r = NULL;
        pthread_join(th[i], &r);
        if (r != NULL)
            rc = -2;
    }
    free(th);
    return rc;
}
