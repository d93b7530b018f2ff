/*
 * kda_oracle.c -- fp64 CPU oracle for Kimi Delta Attention (KDA).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the tests, the package's smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code, header, table or helper with the CUDA
 * library, and it never reads a value produced by the CUDA library.
 *
 * What it computes (plain definition, token by token, one (sequence, head) at a time):
 *
 *   KDA is a gated delta rule whose forget gate acts per key channel
 *   ("per-K-channel exp2(gk)" decay, vllm.cpp PR #110 "chunk_kda prefill AOT port",
 *   commit description; contrasted with GDN's per-head decay in vllm.cpp PR #122
 *   "fold Kimi-Linear onto the shared paged runner", commit body, block B2).
 *   The state of one head is a K x V matrix S (the "[1, nh, hd, hd]" state that is
 *   carried in and out, vllm.cpp PR #113 "paged-incremental decode", commit body).
 *   For token t with key k_t (K), value v_t (V), query q_t (K), natural-log gate
 *   g_t (K) and write strength beta_t (scalar):
 *
 *       S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T
 *       o_t = scale * S_t^T q_t
 *
 *   which this file evaluates in the order
 *       1. S <- Diag(exp g_t) S            (decay each key row c by exp(g_t[c]))
 *       2. u <- S^T k_t                    (read the value stored under k_t)
 *       3. d <- beta_t (v_t - u)           (delta-rule correction)
 *       4. S <- S + k_t d^T                (write)
 *       5. o_t <- scale * S^T q_t          (read out with the updated state)
 *
 *   Prefill runs the steps over every token of each packed sequence
 *   (cu_seqlens), starting from init_state (or zeros), and returns the last S
 *   per sequence.  This is the recurrent form the pages contrast with the
 *   chunked prompt path (PR #110, commit description: "a different reduction
 *   order"); in exact arithmetic both give the same result.
 *
 *   Decode applies the same five steps once per sequence to the state held in
 *   pool slot state_idx[n], in place ("state slots via non_spec_state_indices",
 *   PR #122, block B2; decode advances one token from the carried state, PR #113).
 *
 * Layouts (all row-major, fp64):
 *   q, k : [T, H, K]   v : [T, H, V]   g : [T, H, K]   beta : [T, H]
 *   out  : [T, H, V]   states : [.., H, K, V] (V fastest)
 *
 * Threads: (sequence, head) tasks are independent; they are spread over
 * nthreads POSIX threads.  Each task is evaluated serially, so the result does
 * not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    /* problem */
    int64_t H, K, V;
    const double *q, *k, *v, *g, *beta;
    double scale;
    /* prefill */
    const double *init_state;   /* [N,H,K,V] or NULL */
    const int64_t *cu_seqlens;  /* [N+1] */
    double *final_state;        /* [N,H,K,V] or NULL */
    /* decode */
    double *pool;               /* [S,H,K,V] */
    const int64_t *state_idx;   /* [N] */
    int64_t num_slots;
    /* common */
    double *out;
    int64_t num_tasks;          /* N*H */
    int is_decode;
    /* work distribution */
    pthread_mutex_t lock;
    int64_t next_task;
    int error;
} oracle_job;

/* One token of the recurrence on the K x V state S (row c = key channel). */
static void kda_token_step(double *S, int64_t K, int64_t V,
                           const double *q, const double *k, const double *v,
                           const double *g, double beta, double scale,
                           double *u, double *o)
{
    /* 1. decay */
    for (int64_t c = 0; c < K; ++c) {
        const double a = exp(g[c]);
        for (int64_t j = 0; j < V; ++j) S[c * V + j] *= a;
    }
    /* 2. u = S^T k */
    for (int64_t j = 0; j < V; ++j) u[j] = 0.0;
    for (int64_t c = 0; c < K; ++c)
        for (int64_t j = 0; j < V; ++j) u[j] += S[c * V + j] * k[c];
    /* 3. d = beta (v - u), kept in u */
    for (int64_t j = 0; j < V; ++j) u[j] = beta * (v[j] - u[j]);
    /* 4. S += k d^T */
    for (int64_t c = 0; c < K; ++c)
        for (int64_t j = 0; j < V; ++j) S[c * V + j] += k[c] * u[j];
    /* 5. o = scale S^T q */
    for (int64_t j = 0; j < V; ++j) o[j] = 0.0;
    for (int64_t c = 0; c < K; ++c)
        for (int64_t j = 0; j < V; ++j) o[j] += S[c * V + j] * q[c];
    for (int64_t j = 0; j < V; ++j) o[j] *= scale;
}

static int run_prefill_task(oracle_job *J, int64_t task, double *S, double *u)
{
    const int64_t H = J->H, K = J->K, V = J->V;
    const int64_t n = task / H, h = task % H;
    const int64_t KV = K * V;
    const int64_t bos = J->cu_seqlens[n], eos = J->cu_seqlens[n + 1];
    if (J->init_state) memcpy(S, J->init_state + (n * H + h) * KV, sizeof(double) * KV);
    else memset(S, 0, sizeof(double) * KV);
    for (int64_t t = bos; t < eos; ++t) {
        kda_token_step(S, K, V,
                       J->q + (t * H + h) * K, J->k + (t * H + h) * K,
                       J->v + (t * H + h) * V, J->g + (t * H + h) * K,
                       J->beta[t * H + h], J->scale, u,
                       J->out + (t * H + h) * V);
    }
    if (J->final_state) memcpy(J->final_state + (n * H + h) * KV, S, sizeof(double) * KV);
    return 0;
}

static int run_decode_task(oracle_job *J, int64_t task, double *u)
{
    const int64_t H = J->H, K = J->K, V = J->V;
    const int64_t n = task / H, h = task % H;
    const int64_t slot = J->state_idx[n];
    if (slot < 0 || slot >= J->num_slots) return -1;
    double *S = J->pool + (slot * H + h) * K * V;
    kda_token_step(S, K, V,
                   J->q + (n * H + h) * K, J->k + (n * H + h) * K,
                   J->v + (n * H + h) * V, J->g + (n * H + h) * K,
                   J->beta[n * H + h], J->scale, u, J->out + (n * H + h) * V);
    return 0;
}

static void *worker(void *arg)
{
    oracle_job *J = (oracle_job *)arg;
    double *S = (double *)malloc(sizeof(double) * (size_t)(J->K * J->V));
    double *u = (double *)malloc(sizeof(double) * (size_t)J->V);
    if (!S || !u) {
        pthread_mutex_lock(&J->lock);
        J->error = -2;
        pthread_mutex_unlock(&J->lock);
        free(S); free(u);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int64_t task = J->next_task++;
        pthread_mutex_unlock(&J->lock);
        if (task >= J->num_tasks) break;
        const int rc = J->is_decode ? run_decode_task(J, task, u)
                                    : run_prefill_task(J, task, S, u);
        if (rc) {
            pthread_mutex_lock(&J->lock);
            J->error = rc;
            pthread_mutex_unlock(&J->lock);
        }
    }
    free(S); free(u);
    return NULL;
}

static int run_job(oracle_job *J, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > J->num_tasks) nthreads = (int)(J->num_tasks > 0 ? J->num_tasks : 1);
    pthread_mutex_init(&J->lock, NULL);
    J->next_task = 0;
    J->error = 0;
    pthread_t tids[256];
    int started = 0;
    for (int i = 1; i < nthreads; ++i) {
        if (pthread_create(&tids[started], NULL, worker, J) == 0) ++started;
    }
    worker(J);
    for (int i = 0; i < started; ++i) pthread_join(tids[i], NULL);
    pthread_mutex_destroy(&J->lock);
    return J->error;
}

/*
 * Prefill over packed sequences.  Returns 0, or a negative value on a bad
 * argument (-1) or an allocation failure (-2).
 */
int kda_oracle_prefill(int64_t num_seqs, int64_t H, int64_t K, int64_t V,
                       const double *q, const double *k, const double *v,
                       const double *g, const double *beta, double scale,
                       const double *init_state, const int64_t *cu_seqlens,
                       double *out, double *final_state, int nthreads)
{
    if (num_seqs < 0 || H <= 0 || K <= 0 || V <= 0 || !cu_seqlens) return -1;
    for (int64_t n = 0; n < num_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n] || cu_seqlens[n] < 0) return -1;
    oracle_job J;
    memset(&J, 0, sizeof(J));
    J.H = H; J.K = K; J.V = V;
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.scale = scale;
    J.init_state = init_state; J.cu_seqlens = cu_seqlens; J.final_state = final_state;
    J.out = out; J.num_tasks = num_seqs * H; J.is_decode = 0;
    return run_job(&J, nthreads);
}

/*
 * One decode step for num_seqs sequences; pool slot state_idx[n] of every head
 * is updated in place.  Returns 0, -1 on a bad argument or an index outside
 * [0, num_slots), -2 on an allocation failure.  Slots must be distinct.
 */
int kda_oracle_decode(int64_t num_seqs, int64_t num_slots, int64_t H, int64_t K, int64_t V,
                      const double *q, const double *k, const double *v,
                      const double *g, const double *beta, double scale,
                      double *pool, const int64_t *state_idx, double *out, int nthreads)
{
    if (num_seqs < 0 || num_slots < 0 || H <= 0 || K <= 0 || V <= 0) return -1;
    for (int64_t n = 0; n < num_seqs; ++n)
        if (state_idx[n] < 0 || state_idx[n] >= num_slots) return -1;
    oracle_job J;
    memset(&J, 0, sizeof(J));
    J.H = H; J.K = K; J.V = V;
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.scale = scale;
    J.pool = pool; J.state_idx = state_idx; J.num_slots = num_slots;
    J.out = out; J.num_tasks = num_seqs * H; J.is_decode = 1;
    return run_job(&J, nthreads);
}
