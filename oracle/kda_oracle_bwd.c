/*
 * Kimi Delta Attention (KDA) backward pass -- fp64 CPU ORACLE.
 *
 * TEST INFRASTRUCTURE ONLY.  The slow, plainly written reverse pass that the CUDA
 * backward is checked against.  Only the test suite and the benchmark's CPU-baseline
 * leg may load it.  It shares no code, header, table or helper with the CUDA path,
 * nor with the forward oracle (kda_oracle.c): the forward steps below are written
 * again here.
 *
 * The forward it differentiates (one recurrence per (sequence n, head h); the
 * reading of the FlashKDA pages that the forward oracle documents):
 *
 *   x_t[c]   = exp(A_log[h]) * (g[t,h,c] + dt_bias[h,c])
 *   a_t[c]   = exp(lower_bound * sigmoid(x_t[c]))          decay of key channel c
 *   b_t      = sigmoid(beta_logit[t,h])
 *   S'_t     = Diag(a_t) S_{t-1}
 *   r_t      = S'_t^T k_t ,   d_t = b_t (v_t - r_t)
 *   S_t      = S'_t + k_t d_t^T          (= (I - b k k^T) Diag(a) S_{t-1} + b k v^T)
 *   o_t      = scale * S_t^T q_t
 *
 * Given dO (the gradient of a scalar loss with respect to every o_t) and dS_T (with
 * respect to the final state; zero if absent), the reverse pass takes each step's
 * derivative in the reverse order of the steps above, carrying dS = dL/dS_t:
 *
 *   dS     += scale q_t dO_t^T                   dq_t  = scale S_t dO_t
 *   dd      = dS^T k_t                           dk_t  = dS d_t
 *   dv_t    = b_t dd                             db_t  = dd . (v_t - r_t)
 *   dr      = -b_t dd
 *   dS'     = dS + k_t dr^T                      dk_t += S'_t dr
 *   da_t[c] = sum_j dS'[c,j] S_{t-1}[c,j]        dS    = Diag(a_t) dS'    (= dL/dS_{t-1})
 *
 * then the activations:  dx_t[c] = da_t[c] a_t[c] lower_bound s(1 - s), s = sigmoid(x_t[c]);
 * dg[t,h,c] = dx_t[c] exp(A_log[h]);  ddt_bias[h,c] += dx_t[c] exp(A_log[h]) (= dg);
 * dA_log[h] += sum_c dx_t[c] x_t[c];  dbeta[t,h] = db_t sigmoid'(beta_logit).
 * After the first token dS is the gradient of the initial state.
 *
 * The states S_{t-1} are recomputed from checkpoints taken every 64 tokens of the
 * forward (64 K x V doubles per block), so memory stays bounded at any length.
 *
 * Layouts as in the forward oracle ([rows][H][K|V], states [N][H][K][V], row = key).
 * dA_log and ddt_bias come out per (sequence, head) -- [N][H] and [N][H][K] -- and the
 * caller adds them up over the sequences.  All arithmetic is double (libm exp only);
 * compile with -ffp-contract=off.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define BLOCK 64

typedef struct {
    const double *q, *k, *v, *g, *beta;
    double scale;
    const double *A_log, *dt_bias;
    double lower_bound;
    const double *S0, *dout, *dST;
    double *dq, *dk, *dv, *dg, *dbeta, *dA_log_u, *ddt_u, *dS0;
    const long* seq_start;
    int N, H, K, V;
    const int* heads;
    int n_heads_sel;
    long next_unit;
    pthread_mutex_t lock;
} bwd_job;

static double sigm(double x) { return 1.0 / (1.0 + exp(-x)); }

/* forward quantities of token t (head h): a[c], x[c], b, and S <- step(S) with r and d */
static void fwd_step(const bwd_job* J, long t, int h, double* S, double* a, double* x,
                     double* b, double* r, double* d) {
    const int H = J->H, K = J->K, V = J->V;
    const long rk = (t * H + h) * (long)K, rv = (t * H + h) * (long)V;
    const double eA = exp(J->A_log[h]);
    for (int c = 0; c < K; ++c) {
        x[c] = eA * (J->g[rk + c] + J->dt_bias[(long)h * K + c]);
        a[c] = exp(J->lower_bound * sigm(x[c]));
    }
    *b = sigm(J->beta[t * H + h]);
    for (int c = 0; c < K; ++c)
        for (int j = 0; j < V; ++j) S[(long)c * V + j] *= a[c];
    for (int j = 0; j < V; ++j) r[j] = 0.0;
    for (int c = 0; c < K; ++c)
        for (int j = 0; j < V; ++j) r[j] += S[(long)c * V + j] * J->k[rk + c];
    for (int j = 0; j < V; ++j) d[j] = *b * (J->v[rv + j] - r[j]);
    for (int c = 0; c < K; ++c)
        for (int j = 0; j < V; ++j) S[(long)c * V + j] += J->k[rk + c] * d[j];
}

static void bwd_unit(const bwd_job* J, int n, int h) {
    const int H = J->H, K = J->K, V = J->V;
    const long KV = (long)K * V;
    const long t0 = J->seq_start[n], t1 = J->seq_start[n + 1], L = t1 - t0;
    const long nblk = (L + BLOCK - 1) / BLOCK;
    double* ck = (double*)malloc(sizeof(double) * (size_t)(nblk > 0 ? nblk : 1) * KV);
    double* St = (double*)malloc(sizeof(double) * (size_t)(BLOCK + 1) * KV);  /* S before each token, then after the last */
    double* ab = (double*)malloc(sizeof(double) * (size_t)BLOCK * K);
    double* xb = (double*)malloc(sizeof(double) * (size_t)BLOCK * K);
    double* rb = (double*)malloc(sizeof(double) * (size_t)BLOCK * V);
    double* db_ = (double*)malloc(sizeof(double) * (size_t)BLOCK * V);
    double* bb = (double*)malloc(sizeof(double) * BLOCK);
    double* S = (double*)malloc(sizeof(double) * (size_t)KV);
    double* dS = (double*)malloc(sizeof(double) * (size_t)KV);
    double* dSp = (double*)malloc(sizeof(double) * (size_t)KV);
    double* dd = (double*)malloc(sizeof(double) * (size_t)V);
    double* dr = (double*)malloc(sizeof(double) * (size_t)V);
    double* tmpx = (double*)malloc(sizeof(double) * (size_t)K);
    double* tmpa = (double*)malloc(sizeof(double) * (size_t)K);
    double* tmpr = (double*)malloc(sizeof(double) * (size_t)V);
    double* tmpd = (double*)malloc(sizeof(double) * (size_t)V);
    const long su = (long)n * H + h;

    /* forward: checkpoints of the state before each block */
    if (J->S0) memcpy(S, J->S0 + su * KV, sizeof(double) * KV);
    else memset(S, 0, sizeof(double) * KV);
    for (long bi = 0; bi < nblk; ++bi) {
        memcpy(ck + bi * KV, S, sizeof(double) * KV);
        const long te = t0 + (bi + 1) * BLOCK < t1 ? t0 + (bi + 1) * BLOCK : t1;
        for (long t = t0 + bi * BLOCK; t < te; ++t) {
            double bt;
            fwd_step(J, t, h, S, tmpa, tmpx, &bt, tmpr, tmpd);
        }
    }

    /* reverse */
    if (J->dST) memcpy(dS, J->dST + su * KV, sizeof(double) * KV);
    else memset(dS, 0, sizeof(double) * KV);
    double dA = 0.0;
    double* ddt = J->ddt_u + su * K;
    for (int c = 0; c < K; ++c) ddt[c] = 0.0;
    const double eA = exp(J->A_log[h]);
    for (long bi = nblk - 1; bi >= 0; --bi) {
        const long ts = t0 + bi * BLOCK;
        const long te = ts + BLOCK < t1 ? ts + BLOCK : t1;
        const int len = (int)(te - ts);
        memcpy(St, ck + bi * KV, sizeof(double) * KV);
        for (int i = 0; i < len; ++i) {
            memcpy(St + (long)(i + 1) * KV, St + (long)i * KV, sizeof(double) * KV);
            fwd_step(J, ts + i, h, St + (long)(i + 1) * KV, ab + (long)i * K, xb + (long)i * K,
                     bb + i, rb + (long)i * V, db_ + (long)i * V);
        }
        for (int i = len - 1; i >= 0; --i) {
            const long t = ts + i;
            const long rk = (t * H + h) * (long)K, rv = (t * H + h) * (long)V;
            const double* Sprev = St + (long)i * KV;       /* S_{t-1} */
            const double* Snow = St + (long)(i + 1) * KV;  /* S_t     */
            const double* a = ab + (long)i * K;
            const double* x = xb + (long)i * K;
            const double* r = rb + (long)i * V;
            const double* d = db_ + (long)i * V;
            const double b = bb[i];
            const double* qt = J->q + rk;
            const double* kt = J->k + rk;
            const double* vt = J->v + rv;
            const double* dot = J->dout + rv;
            /* dS += scale q dO^T ; dq = scale S_t dO */
            for (int c = 0; c < K; ++c) {
                double acc = 0.0;
                for (int j = 0; j < V; ++j) {
                    dS[(long)c * V + j] += J->scale * qt[c] * dot[j];
                    acc += Snow[(long)c * V + j] * dot[j];
                }
                J->dq[rk + c] = J->scale * acc;
            }
            /* dd = dS^T k ; dk = dS d */
            for (int j = 0; j < V; ++j) dd[j] = 0.0;
            for (int c = 0; c < K; ++c)
                for (int j = 0; j < V; ++j) dd[j] += dS[(long)c * V + j] * kt[c];
            for (int c = 0; c < K; ++c) {
                double acc = 0.0;
                for (int j = 0; j < V; ++j) acc += dS[(long)c * V + j] * d[j];
                J->dk[rk + c] = acc;
            }
            /* dv, db, dr */
            double dbt = 0.0;
            for (int j = 0; j < V; ++j) {
                J->dv[rv + j] = b * dd[j];
                dbt += dd[j] * (vt[j] - r[j]);
                dr[j] = -b * dd[j];
            }
            /* dS' = dS + k dr^T ; dk += S' dr ; da ; dS = Diag(a) dS' */
            for (int c = 0; c < K; ++c) {
                double acc = 0.0, da = 0.0;
                for (int j = 0; j < V; ++j) {
                    const long e = (long)c * V + j;
                    dSp[e] = dS[e] + kt[c] * dr[j];
                    acc += a[c] * Sprev[e] * dr[j];
                    da += dSp[e] * Sprev[e];
                }
                J->dk[rk + c] += acc;
                for (int j = 0; j < V; ++j) dS[(long)c * V + j] = a[c] * dSp[(long)c * V + j];
                /* the gate: a = exp(lb * sigmoid(x)) */
                const double s = sigm(x[c]);
                const double dx = da * a[c] * J->lower_bound * s * (1.0 - s);
                J->dg[rk + c] = dx * eA;
                ddt[c] += dx * eA;
                dA += dx * x[c];
            }
            const double sb = sigm(J->beta[t * H + h]);
            J->dbeta[t * H + h] = dbt * sb * (1.0 - sb);
        }
    }
    if (J->dS0) memcpy(J->dS0 + su * KV, dS, sizeof(double) * KV);
    J->dA_log_u[su] = dA;

    free(ck); free(St); free(ab); free(xb); free(rb); free(db_); free(bb);
    free(S); free(dS); free(dSp); free(dd); free(dr); free(tmpx); free(tmpa); free(tmpr);
    free(tmpd);
}

static void* bwd_worker(void* arg) {
    bwd_job* J = (bwd_job*)arg;
    const long units = (long)J->N * J->n_heads_sel;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        long u = J->next_unit++;
        pthread_mutex_unlock(&J->lock);
        if (u >= units) break;
        int n = (int)(u / J->n_heads_sel);
        int hs = (int)(u % J->n_heads_sel);
        bwd_unit(J, n, J->heads ? J->heads[hs] : hs);
    }
    return NULL;
}

/* heads / n_heads_sel: optional subset of heads (NULL = all); entries of the other
 * heads are left untouched. */
int kda_oracle_bwd(const double* q, const double* k, const double* v, const double* g,
                   const double* beta_logit, double scale, const double* A_log,
                   const double* dt_bias, double lower_bound, const double* S0,
                   const double* dout, const double* dST, double* dq, double* dk, double* dv,
                   double* dg, double* dbeta, double* dA_log_u, double* ddt_u, double* dS0,
                   const long* seq_start, int N, int H, int K, int V, const int* heads,
                   int n_heads_sel, int n_threads) {
    if (N < 0 || H <= 0 || K <= 0 || V <= 0) return -1;
    for (int n = 0; n < N; ++n)
        if (seq_start[n + 1] < seq_start[n]) return -2;
    bwd_job J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta_logit; J.scale = scale;
    J.A_log = A_log; J.dt_bias = dt_bias; J.lower_bound = lower_bound;
    J.S0 = S0; J.dout = dout; J.dST = dST;
    J.dq = dq; J.dk = dk; J.dv = dv; J.dg = dg; J.dbeta = dbeta;
    J.dA_log_u = dA_log_u; J.ddt_u = ddt_u; J.dS0 = dS0;
    J.seq_start = seq_start; J.N = N; J.H = H; J.K = K; J.V = V;
    J.heads = heads; J.n_heads_sel = heads ? n_heads_sel : H;
    long units = (long)N * J.n_heads_sel;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > units) n_threads = (int)(units > 0 ? units : 1);
    J.next_unit = 0;
    pthread_mutex_init(&J.lock, NULL);
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
    for (int i = 0; i < n_threads; ++i) pthread_create(&th[i], NULL, bwd_worker, &J);
    for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return 0;
}
