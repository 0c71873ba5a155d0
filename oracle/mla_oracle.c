/*
 * mla_oracle.c -- the fp64 CPU oracle for one decode step of gated multi-head
 * latent attention, the exact-attention layer that the pages interleave with
 * the incremental linear attention.
 *
 * TEST INFRASTRUCTURE.  Only the tests and the benchmark's CPU-baseline leg
 * may load this file's library.  It shares no code, header, table or helper
 * with the CUDA library, and never calls it.
 *
 * What the pages say, and the reading taken here.  The layer "compresses the
 * Key/Value projections into a low-dimensional latent space", so that the
 * cache holds one small latent vector per token instead of per-head keys and
 * values, keeps exact (softmax) attention for precise retrieval, and adds a
 * gate ("Trillion-Parameter MoE Multimodal LLMs: How to Evaluate the New
 * Generation", section 2.1; "How to Think About Trillion-Parameter Sparse
 * Multimodal LLMs", section 2.3; "How Large-Scale MoE Multimodal LLMs Are
 * Evolving: Architecture, Training, and Engineering Practices", section 2).
 * The pages give no equations, so the plainest reading is:
 *
 *   latent        c_t = W_dkv x_t                          (cached, d_c values)
 *   per head h    k_{t,h} = W_uk,h c_t,  v_{t,h} = W_uv,h c_t      (d_h values)
 *   score         s_{t,h} = scale * q_h . k_{t,h} = scale * (W_uk,h^T q_h) . c_t
 *   attention     o_h = sum_t softmax_t(s_{.,h}) v_{t,h} = W_uv,h sum_t p_{t,h} c_t
 *   gate          y_h = sigmoid(z_h) * o_h       (elementwise, z_h = W_g,h x)
 *
 * The decode step takes the query already multiplied by W_uk,h^T (q_abs, d_c
 * values per head: the key projection absorbed into the query, so keys are
 * never formed), the latent cache, the per-sequence cache lengths, W_uv and the
 * gate's pre-activation z; it returns y.  Here the softmax is evaluated as its
 * definition, with the row maximum subtracted first (an identity of the
 * softmax) so that no exponential overflows, then the weighted sum of latents,
 * the value up-projection and the gate.  A sequence of length 0 has no terms:
 * its output is zero.
 *
 * Layouts: q_abs [N][H][dc], ckv [N][Lmax][dc], seqlens [N], w_uv [H][dh][dc],
 * gate [N][H][dh], out [N][H][dh].  Inputs are float32 arrays (bf16 inputs
 * widened exactly by the caller); all arithmetic is fp64.
 *
 * Parity status: pinned by the CPU tests -- agreement with attention written
 * out over explicitly up-projected keys and values (no absorption), the
 * one-token and identical-latents closed forms, the uniform average for a zero
 * query, a dominant score far beyond exp's range, the masking of cache rows
 * past the length, the gate's limits, and planted mistakes.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* One (sequence, head).  qa [dc]; ckv [len][dc]; wuv [dh][dc]; z [dh]; out [dh];
 * scratch s [len], ol [dc]. */
static void mla_one(const float *qa, const float *ckv, int64_t len, const float *wuv,
                    const float *z, double scale, double *out, int dc, int dh, double *s,
                    double *ol)
{
    int c, j;
    int64_t t;
    for (c = 0; c < dc; ++c) ol[c] = 0.0;
    if (len > 0) {
        double m = -INFINITY, l = 0.0;
        for (t = 0; t < len; ++t) {
            double acc = 0.0;
            for (c = 0; c < dc; ++c) acc += (double)qa[c] * (double)ckv[t * dc + c];
            s[t] = scale * acc;
            if (s[t] > m) m = s[t];
        }
        for (t = 0; t < len; ++t) {
            const double p = exp(s[t] - m);
            l += p;
            for (c = 0; c < dc; ++c) ol[c] += p * (double)ckv[t * dc + c];
        }
        for (c = 0; c < dc; ++c) ol[c] /= l;
    }
    for (j = 0; j < dh; ++j) {
        double o = 0.0;
        for (c = 0; c < dc; ++c) o += (double)wuv[(int64_t)j * dc + c] * ol[c];
        out[j] = sigmoid((double)z[j]) * o;
    }
}

struct mla_job {
    const float *q_abs, *ckv, *w_uv, *gate;
    const int *seqlens;
    double scale;
    double *out;
    int N, H, Lmax, dc, dh;
    int64_t next, end;
    pthread_mutex_t *mu;
    int err;
};

static void *mla_worker(void *arg)
{
    struct mla_job *J = (struct mla_job *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)(J->Lmax > 0 ? J->Lmax : 1));
    double *ol = (double *)malloc(sizeof(double) * (size_t)J->dc);
    if (!s || !ol) {
        free(s);
        free(ol);
        pthread_mutex_lock(J->mu);
        J->err = 1;
        pthread_mutex_unlock(J->mu);
        return NULL;
    }
    for (;;) {
        int64_t item;
        pthread_mutex_lock(J->mu);
        item = J->next < J->end ? J->next++ : -1;
        pthread_mutex_unlock(J->mu);
        if (item < 0) break;
        {
            const int64_t n = item / J->H, h = item % J->H;
            int64_t len = J->seqlens[n];
            if (len < 0) len = 0;
            if (len > J->Lmax) len = J->Lmax;
            mla_one(J->q_abs + (n * J->H + h) * J->dc, J->ckv + n * (int64_t)J->Lmax * J->dc, len,
                    J->w_uv + h * (int64_t)J->dh * J->dc, J->gate + (n * J->H + h) * J->dh,
                    J->scale, J->out + (n * J->H + h) * J->dh, J->dc, J->dh, s, ol);
        }
    }
    free(s);
    free(ol);
    return NULL;
}

/* Returns 0, or 1 for bad arguments or a failed allocation.  Lengths are
 * clamped into [0, Lmax]. */
int gdr_oracle_mla_decode(const float *q_abs, const float *ckv, const int *seqlens,
                          const float *w_uv, const float *gate, double scale, double *out,
                          int N, int H, int Lmax, int dc, int dh, int nthreads)
{
    struct mla_job J;
    pthread_mutex_t mu = PTHREAD_MUTEX_INITIALIZER;
    pthread_t *th;
    int i, nt;
    if (N < 0 || H < 0 || Lmax < 0 || dc <= 0 || dh <= 0) return 1;
    if ((int64_t)N * H == 0) return 0;
    J.q_abs = q_abs;
    J.ckv = ckv;
    J.w_uv = w_uv;
    J.gate = gate;
    J.seqlens = seqlens;
    J.scale = scale;
    J.out = out;
    J.N = N;
    J.H = H;
    J.Lmax = Lmax;
    J.dc = dc;
    J.dh = dh;
    J.next = 0;
    J.end = (int64_t)N * H;
    J.mu = &mu;
    J.err = 0;
    nt = nthreads < 1 ? 1 : nthreads;
    if (nt > J.end) nt = (int)J.end;
    th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    if (!th) return 1;
    for (i = 0; i < nt; ++i) pthread_create(&th[i], NULL, mla_worker, &J);
    for (i = 0; i < nt; ++i) pthread_join(th[i], NULL);
    free(th);
    return J.err;
}
