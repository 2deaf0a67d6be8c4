/*
 * Kimi Delta Attention (KDA) forward pass -- fp64 CPU ORACLE.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plainly written
 * definition that the CUDA library is checked against.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (one independent recurrence per (sequence n, head h)):
 *
 *   gate      gl[t,c]  = lower_bound * sigmoid(exp(A_log[h]) * (g[t,h,c] + dt_bias[h,c]))
 *             alpha[c] = exp(gl[t,c])                      (natural-log decay, c = 0..K-1)
 *   beta      b_t      = sigmoid(beta_logit[t,h])
 *   state     S_t      = (I - b_t k_t k_t^T) Diag(alpha_t) S_{t-1} + b_t k_t v_t^T   (S is K x V)
 *   output    o_t      = scale * S_t^T q_t                 (the state AFTER the update at t)
 *
 * Sources (web pages on Moonshot AI's FlashKDA release):
 *   - "Moonshot AI Rilis FlashKDA" (captivela.com), paragraphs on the forward
 *     pass inputs (q, k, v, pre-activation gate g, beta logits, scale, A_log,
 *     dt_bias, lower_bound), sigmoid applied to beta inside the kernel, and the
 *     optional initial / final recurrent states; KDA is Gated DeltaNet with
 *     channel-wise gating.
 *   - "Moonshot AI Open-Sources FlashKDA" (alphasignal.ai), section "Why KDA?":
 *     channel-by-channel gating of what is written to and kept in memory.
 *   The pages describe the recurrence in words only (a gated delta rule whose
 *   decay is per channel) and print no equation.  The form above is the
 *   gated delta rule with Diag(alpha) in place of Gated DeltaNet's scalar
 *   decay; that o_t reads the state after the update at t is part of that
 *   reading.  The gate formula is a reading too (the pages name A_log,
 *   dt_bias and lower_bound but print no formula): lower_bound is taken as
 *   the lower bound of the per-token log-decay, which the sigmoid form keeps
 *   strictly inside (lower_bound, 0).
 *
 * The update is evaluated in the algebraically equal order
 *   S' = Diag(alpha) S ;  S = S' + b k (v - S'^T k)^T
 * which is (I - b k k^T) S' + b k v^T expanded once.
 *
 * Layouts (row-major, element strides):
 *   q, k, g   : [rows][H][K]      v, out : [rows][H][V]     beta : [rows][H]
 *   A_log [H]; dt_bias [H][K]; states [N][H][K][V] (row = K index, col = V index)
 *   seq_start [N+1] : token rows of sequence n are seq_start[n] .. seq_start[n+1]-1
 *
 * All arithmetic is double; transcendental calls are libm exp only.
 * Compile with -O2 -ffp-contract=off (no fast-math) so results do not depend
 * on FMA contraction.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ---- gate: per-channel natural-log decay -------------------------------- */

static double oracle_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

static double oracle_gate_one(double g, double A_log, double dt_bias, double lower_bound) {
    return lower_bound * oracle_sigmoid(exp(A_log) * (g + dt_bias));
}

/* out[r][h][c] = log-decay for every row r, head h, channel c. */
void kda_oracle_gate(const double* g, const double* A_log, const double* dt_bias,
                     double lower_bound, double* out, long rows, int H, int K) {
    for (long r = 0; r < rows; ++r)
        for (int h = 0; h < H; ++h)
            for (int c = 0; c < K; ++c) {
                long i = (r * H + h) * (long)K + c;
                out[i] = oracle_gate_one(g[i], A_log[h], dt_bias[(long)h * K + c], lower_bound);
            }
}

/* ---- one (sequence, head) recurrence ------------------------------------ */

typedef struct {
    const double *q, *k, *v;
    const double *g;          /* pre-activation gate (gate mode) or NULL */
    const double *log_alpha;  /* natural-log decay (raw mode) or NULL     */
    const double *beta;       /* logits (gate mode) or post-sigmoid (raw) */
    double scale;
    const double *A_log, *dt_bias;
    double lower_bound;
    const double* S0;
    double* S_final;
    double* out;
    const long* seq_start;
    int N, H, K, V;
    const int* heads;
    int n_heads_sel;
    /* work queue */
    long next_unit;
    pthread_mutex_t lock;
} oracle_job;

static void oracle_unit(const oracle_job* J, int n, int h, double* S, double* a,
                        double* p) {
    const int H = J->H, K = J->K, V = J->V;
    const long unitKV = (long)K * V;
    if (J->S0)
        memcpy(S, J->S0 + ((long)n * H + h) * unitKV, sizeof(double) * unitKV);
    else
        memset(S, 0, sizeof(double) * unitKV);

    for (long t = J->seq_start[n]; t < J->seq_start[n + 1]; ++t) {
        const long rk = (t * H + h) * (long)K;  /* row offset in [rows][H][K] */
        const long rv = (t * H + h) * (long)V;  /* row offset in [rows][H][V] */
        const double* kt = J->k + rk;
        const double* qt = J->q + rk;
        const double* vt = J->v + rv;

        /* decay factors alpha_t[c] and write strength b_t */
        double b;
        if (J->g) {
            for (int c = 0; c < K; ++c)
                a[c] = exp(oracle_gate_one(J->g[rk + c], J->A_log[h],
                                           J->dt_bias[(long)h * K + c], J->lower_bound));
            b = oracle_sigmoid(J->beta[t * H + h]);
        } else {
            for (int c = 0; c < K; ++c) a[c] = exp(J->log_alpha[rk + c]);
            b = J->beta[t * H + h];
        }

        /* S' = Diag(alpha) S : row c of S is scaled by alpha[c] */
        for (int c = 0; c < K; ++c)
            for (int j = 0; j < V; ++j) S[(long)c * V + j] *= a[c];

        /* p = S'^T k */
        for (int j = 0; j < V; ++j) p[j] = 0.0;
        for (int c = 0; c < K; ++c)
            for (int j = 0; j < V; ++j) p[j] += S[(long)c * V + j] * kt[c];

        /* S = S' + b k (v - p)^T */
        for (int j = 0; j < V; ++j) p[j] = b * (vt[j] - p[j]);
        for (int c = 0; c < K; ++c)
            for (int j = 0; j < V; ++j) S[(long)c * V + j] += kt[c] * p[j];

        /* o_t = scale * S^T q */
        double* ot = J->out + rv;
        for (int j = 0; j < V; ++j) ot[j] = 0.0;
        for (int c = 0; c < K; ++c)
            for (int j = 0; j < V; ++j) ot[j] += S[(long)c * V + j] * qt[c];
        for (int j = 0; j < V; ++j) ot[j] *= J->scale;
    }

    if (J->S_final)
        memcpy(J->S_final + ((long)n * H + h) * unitKV, S, sizeof(double) * unitKV);
}

static void* oracle_worker(void* arg) {
    oracle_job* J = (oracle_job*)arg;
    const long units = (long)J->N * J->n_heads_sel;
    double* S = (double*)malloc(sizeof(double) * (size_t)J->K * J->V);
    double* a = (double*)malloc(sizeof(double) * (size_t)J->K);
    double* p = (double*)malloc(sizeof(double) * (size_t)J->V);
    for (;;) {
        pthread_mutex_lock(&J->lock);
        long u = J->next_unit++;
        pthread_mutex_unlock(&J->lock);
        if (u >= units) break;
        int n = (int)(u / J->n_heads_sel);
        int hs = (int)(u % J->n_heads_sel);
        int h = J->heads ? J->heads[hs] : hs;
        oracle_unit(J, n, h, S, a, p);
    }
    free(S);
    free(a);
    free(p);
    return NULL;
}

static int oracle_run(oracle_job* J, int n_threads) {
    if (J->N < 0 || J->H <= 0 || J->K <= 0 || J->V <= 0) return -1;
    if (!J->heads) J->n_heads_sel = J->H;
    for (int n = 0; n < J->N; ++n)
        if (J->seq_start[n + 1] < J->seq_start[n]) return -2;
    long units = (long)J->N * J->n_heads_sel;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > units) n_threads = (int)(units > 0 ? units : 1);
    J->next_unit = 0;
    pthread_mutex_init(&J->lock, NULL);
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
    for (int i = 0; i < n_threads; ++i) pthread_create(&th[i], NULL, oracle_worker, J);
    for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J->lock);
    return 0;
}

/* Full forward: gate and beta activations applied here.
 * heads / n_heads_sel: optional subset of heads to evaluate (NULL = all);
 * outputs of heads outside the subset are left untouched. */
int kda_oracle_fwd(const double* q, const double* k, const double* v, const double* g,
                   const double* beta_logit, double scale, const double* A_log,
                   const double* dt_bias, double lower_bound, const double* S0,
                   double* S_final, double* out, const long* seq_start, int N, int H,
                   int K, int V, const int* heads, int n_heads_sel, int n_threads) {
    oracle_job J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.g = g; J.log_alpha = NULL; J.beta = beta_logit;
    J.scale = scale; J.A_log = A_log; J.dt_bias = dt_bias; J.lower_bound = lower_bound;
    J.S0 = S0; J.S_final = S_final; J.out = out; J.seq_start = seq_start;
    J.N = N; J.H = H; J.K = K; J.V = V; J.heads = heads; J.n_heads_sel = n_heads_sel;
    return oracle_run(&J, n_threads);
}

/* Raw recurrence: the caller gives the natural-log decay [rows][H][K] and the
 * post-activation write strength beta [rows][H] directly (no gate, no sigmoid). */
int kda_oracle_recurrence(const double* q, const double* k, const double* v,
                          const double* log_alpha, const double* beta, double scale,
                          const double* S0, double* S_final, double* out,
                          const long* seq_start, int N, int H, int K, int V,
                          const int* heads, int n_heads_sel, int n_threads) {
    oracle_job J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.g = NULL; J.log_alpha = log_alpha; J.beta = beta;
    J.scale = scale; J.S0 = S0; J.S_final = S_final; J.out = out; J.seq_start = seq_start;
    J.N = N; J.H = H; J.K = K; J.V = V; J.heads = heads; J.n_heads_sel = n_heads_sel;
    return oracle_run(&J, n_threads);
}
