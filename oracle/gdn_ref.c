/*
 * fp64 CPU oracle of the gated delta rule (Gated DeltaNet), token by token.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the package's smoke check and
 * the benchmark's CPU-baseline leg may load this library. It shares no code,
 * header or constant with the CUDA path.
 *
 * What it computes (the recurrence the chunked kernels of the "WarpDrive"
 * page, kernels 3-5, are a blocked form of): for every sequence (b, h), with
 * the state S a K x V matrix,
 *
 *     S_0   = h0 (or 0)
 *     a_t   = exp(gamma_t)
 *     S    <- a_t * S                          (decay first)
 *     d_t   = beta_t * (v_t - S^T k_t)         (read the decayed state)
 *     S    <- S + k_t d_t^T                    (delta-rule write)
 *     o_t   = scale * S^T q_t                  (query the updated state)
 *     h_final = S_T
 *
 * The same operation order (decay, read, write, query the updated state)
 * appears in the per-token update of the vLLM KDA decode kernel page
 * (method `update`).
 *
 * gamma_t is the per-token log-decay. The caller passes g, the cumulative sum
 * of gamma restarted at every `chunk` tokens (the form the chunked kernels
 * consume), so gamma_t = g_t - g_{t-1} inside a chunk and gamma_t = g_t at the
 * first token of a chunk. The difference of two fp32 values is exact in fp64.
 *
 * Per-channel decay (the KDA variant: the decay is a K-vector, one factor per
 * row of S, as in the "KdaSplit" decode kernel page, where each state row is
 * scaled by its own decay before the read): with per_channel set, g is
 * [B,T,H,K], gamma_t is a K-vector read from g the same way, and the decay
 * step is S[i, :] <- exp(gamma_t[i]) * S[i, :]. Everything else is unchanged.
 *
 * Layout: q, k [B,T,H,K]; v, o [B,T,H,V]; g, beta [B,T,H] (g [B,T,H,K] with
 * per_channel); h0, h_final [B,H,K,V]; all fp64, contiguous. h0 may be NULL
 * (zero state), h_final may be NULL (not written).
 *
 * Optional exports (NULL = not written), used to check the stages of a chunked
 * implementation against the recurrence:
 *   h_chunks [B,NT,H,K,V]  the state entering each chunk (NT = ceil(T/chunk))
 *   delta    [B,T,H,V]     the per-token correction d_t above
 *
 * Threads: a static interleaved split of the B*H independent sequences over
 * `nthreads` POSIX threads (nthreads <= 1 runs inline).
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int B, T, H, K, V, chunk, per_channel;
    const double *q, *k, *v, *g, *beta;
    double scale;
    const double *h0;
    double *o, *h_final, *h_chunks, *delta;
    int tid, nthreads;
    int status;
} job_t;

static void run_sequence(const job_t *j, int b, int h, double *S, double *d)
{
    const int T = j->T, H = j->H, K = j->K, V = j->V;
    const size_t kv = (size_t)K * V;
    if (j->h0)
        memcpy(S, j->h0 + ((size_t)b * H + h) * kv, kv * sizeof(double));
    else
        memset(S, 0, kv * sizeof(double));

    for (int t = 0; t < T; ++t) {
        const size_t row = (size_t)b * T * H + (size_t)t * H + h;   /* (b,t,h) */
        const double *qt = j->q + row * K;
        const double *kt = j->k + row * K;
        const double *vt = j->v + row * V;
        const double bt = j->beta[row];

        if (j->h_chunks && t % j->chunk == 0) {
            const int NT = (T + j->chunk - 1) / j->chunk;
            const size_t slot = ((size_t)b * NT + t / j->chunk) * H + h;
            memcpy(j->h_chunks + slot * kv, S, kv * sizeof(double));
        }
        if (!j->per_channel) {
            const double gt = j->g[row];
            const double gamma = (t % j->chunk == 0) ? gt : gt - j->g[row - H];
            const double a = exp(gamma);
            for (size_t e = 0; e < kv; ++e)
                S[e] *= a;
        } else {
            /* row i of S decays by its own channel's factor */
            const double *gk = j->g + row * K;
            for (int i = 0; i < K; ++i) {
                /* inside a chunk: minus the same channel of token t - 1 (row - H) */
                const double gamma_i =
                    (t % j->chunk == 0) ? gk[i] : gk[i] - j->g[(row - H) * K + i];
                const double ai = exp(gamma_i);
                double *Si = S + (size_t)i * V;
                for (int c = 0; c < V; ++c)
                    Si[c] *= ai;
            }
        }
        for (int c = 0; c < V; ++c) {
            double r = 0.0;
            for (int i = 0; i < K; ++i)
                r += S[(size_t)i * V + c] * kt[i];
            d[c] = bt * (vt[c] - r);
        }
        if (j->delta)
            memcpy(j->delta + row * V, d, (size_t)V * sizeof(double));
        for (int i = 0; i < K; ++i) {
            double *Si = S + (size_t)i * V;
            for (int c = 0; c < V; ++c)
                Si[c] += kt[i] * d[c];
        }
        double *ot = j->o + row * V;
        for (int c = 0; c < V; ++c) {
            double r = 0.0;
            for (int i = 0; i < K; ++i)
                r += S[(size_t)i * V + c] * qt[i];
            ot[c] = j->scale * r;
        }
    }
    if (j->h_final)
        memcpy(j->h_final + ((size_t)b * H + h) * kv, S, kv * sizeof(double));
}

static void *worker(void *arg)
{
    job_t *j = (job_t *)arg;
    double *S = (double *)malloc((size_t)j->K * j->V * sizeof(double));
    double *d = (double *)malloc((size_t)j->V * sizeof(double));
    if (!S || !d) {
        j->status = 2;
        free(S);
        free(d);
        return NULL;
    }
    for (int s = j->tid; s < j->B * j->H; s += j->nthreads)
        run_sequence(j, s / j->H, s % j->H, S, d);
    free(S);
    free(d);
    return NULL;
}

/* Returns 0 on success, 1 on bad arguments, 2 on host allocation failure.
 * Sequences whose thread could not be started run on the calling thread. */
int gdn_oracle_forward_pc(int B, int T, int H, int K, int V, int chunk, int per_channel,
                          const double *q, const double *k, const double *v,
                          const double *g, const double *beta, double scale,
                          const double *h0, double *o, double *h_final,
                          double *h_chunks, double *delta, int nthreads)
{
    if (B <= 0 || T < 0 || H <= 0 || K <= 0 || V <= 0 || chunk <= 0)
        return 1;
    if (!q || !k || !v || !g || !beta || !o)
        return 1;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > B * H)
        nthreads = B * H;

    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return 2;
    }
    for (int i = 0; i < nthreads; ++i) {
        job_t *j = &jobs[i];
        j->B = B; j->T = T; j->H = H; j->K = K; j->V = V; j->chunk = chunk;
        j->per_channel = per_channel;
        j->q = q; j->k = k; j->v = v; j->g = g; j->beta = beta; j->scale = scale;
        j->h0 = h0; j->o = o; j->h_final = h_final;
        j->h_chunks = h_chunks; j->delta = delta;
        j->tid = i; j->nthreads = nthreads; j->status = 0;
    }
    int rc = 0, started = 0;
    if (nthreads > 1)
        while (started < nthreads &&
               pthread_create(&th[started], NULL, worker, &jobs[started]) == 0)
            ++started;
    for (int i = started; i < nthreads; ++i)
        worker(&jobs[i]);
    for (int i = 0; i < started; ++i)
        pthread_join(th[i], NULL);
    for (int i = 0; i < nthreads; ++i)
        if (jobs[i].status)
            rc = jobs[i].status;
    free(jobs);
    free(th);
    return rc;
}

int gdn_oracle_forward_ex(int B, int T, int H, int K, int V, int chunk,
                          const double *q, const double *k, const double *v,
                          const double *g, const double *beta, double scale,
                          const double *h0, double *o, double *h_final,
                          double *h_chunks, double *delta, int nthreads)
{
    return gdn_oracle_forward_pc(B, T, H, K, V, chunk, 0, q, k, v, g, beta, scale, h0, o,
                                 h_final, h_chunks, delta, nthreads);
}

int gdn_oracle_forward(int B, int T, int H, int K, int V, int chunk,
                       const double *q, const double *k, const double *v,
                       const double *g, const double *beta, double scale,
                       const double *h0, double *o, double *h_final, int nthreads)
{
    return gdn_oracle_forward_ex(B, T, H, K, V, chunk, q, k, v, g, beta, scale, h0, o,
                                 h_final, NULL, NULL, nthreads);
}
