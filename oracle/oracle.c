/*
 * oracle.c -- plain, slow fp64 CPU reference for the gated delta rule.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark load this file's library. The CUDA library never includes, links or calls
 * it, and this file uses nothing of the CUDA library: the two share no code.
 *
 * Sources (web pages; cited by title and section):
 *   [RFC]  "RFC: HyperParallel Linear Attention Context Parallel", section 2.1 (the
 *          per-token recurrence) and section 2.2 (the affine summary H_out = M@H_in + S
 *          and its compose rule).
 *   [ART]  "Context Parallelism in ART", section 08 "Gated DeltaNet context
 *          parallelism", sub-sections "First parallelize within a GPU" (chunk
 *          equations) and "Then parallelize across GPUs" (summary, compose, scan).
 *
 * Conventions. One (b,h) head has a K x V state H. Inputs are float arrays holding the
 * values exactly as stored (bf16 inputs arrive already rounded); every operation here is
 * done in double. Layouts (row-major, contiguous):
 *   q, k : [B, T, H, K]     v, o : [B, T, H, V]     g, beta : [B, T, H]
 *   states h0, h_final : [B, H, K, V]
 *   summaries M : [nseg, B, H, K, K],  S : [nseg, B, H, K, V]
 *
 * Readings of the pages that this file takes (each listed in the design notes):
 *   - the recurrence reads the un-decayed state H_{t-1} ([RFC] 2.1), so the per-token
 *     transition is exp(g_t) I - beta_t k_t k_t^T; with decay_first set, every function
 *     takes the other reading ([ART] 08 "What a GDN token does to the state"; [KDA] "KDA
 *     Chunk Backward -- TPU/Pallas Kernel Design" 1.2): the read sees exp(g_t) H_{t-1}, the
 *     transition is exp(g_t) (I - beta_t k_t k_t^T), and the chunk form uses the inclusive
 *     cumulative gate G_i where the default uses the exclusive Gx_i (in P and Kr);
 *   - g is a natural-log decay (exp(g_t)); no query scale;
 *   - segments are contiguous, equal length, in token order; segment 0 starts from h0.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------------------ */
/* a tiny work queue over "units": each thread takes the next unit index atomically      */
/* ------------------------------------------------------------------------------------ */
typedef void (*unit_fn)(void* ctx, long unit);
typedef struct {
    unit_fn fn;
    void* ctx;
    long n_units;
    long next;
    pthread_mutex_t lock;
} pool_t;

static void* pool_worker(void* arg) {
    pool_t* p = (pool_t*)arg;
    for (;;) {
        pthread_mutex_lock(&p->lock);
        long u = p->next++;
        pthread_mutex_unlock(&p->lock);
        if (u >= p->n_units) break;
        p->fn(p->ctx, u);
    }
    return NULL;
}

static int resolve_threads(int nthreads) {
    if (nthreads > 0) return nthreads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static void run_units(unit_fn fn, void* ctx, long n_units, int nthreads) {
    pool_t p;
    p.fn = fn;
    p.ctx = ctx;
    p.n_units = n_units;
    p.next = 0;
    pthread_mutex_init(&p.lock, NULL);
    int nt = resolve_threads(nthreads);
    if (nt > n_units) nt = (int)n_units;
    if (nt <= 1) {
        pool_worker(&p);
    } else {
        pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nt);
        for (int i = 0; i < nt; ++i) pthread_create(&th[i], NULL, pool_worker, &p);
        for (int i = 0; i < nt; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&p.lock);
}

int oracle_num_threads(int nthreads) { return resolve_threads(nthreads); }

/* ------------------------------------------------------------------------------------ */
/* 1. Per-token recurrence ([RFC] 2.1), literally:                                        */
/*      residual_t = beta_t * (v_t - k_t @ H_{t-1})                                      */
/*      H_t        = exp(g_t) * H_{t-1} + outer(k_t, residual_t)                          */
/*      o_t        = q_t @ H_t                                                           */
/* Column v of H only ever meets column v of the value vectors, so the columns are       */
/* independent recurrences; a work unit is one (b, h, block of columns).                 */
/* ------------------------------------------------------------------------------------ */
typedef struct {
    int B, T, H, K, V, seg_len, col_block;
    const float *q, *k, *v, *g, *beta, *h0;
    double *o, *h_final, *H_in;
    int decay_first;   /* read exp(g_t) H_{t-1} instead of H_{t-1} (the other reading) */
} rec_ctx;

static void rec_unit(void* vctx, long unit) {
    const rec_ctx* c = (const rec_ctx*)vctx;
    const int K = c->K, V = c->V, H = c->H, T = c->T;
    const int nblk = (V + c->col_block - 1) / c->col_block;
    const int blk = (int)(unit % nblk);
    const long bh = unit / nblk;
    const int b = (int)(bh / H), h = (int)(bh % H);
    const int c0 = blk * c->col_block;
    const int nc = (c0 + c->col_block <= V) ? c->col_block : V - c0;

    double* S = (double*)malloc(sizeof(double) * (size_t)K * (size_t)nc); /* S[kk][cc] */
    double* kt = (double*)malloc(sizeof(double) * (size_t)K);
    double* qt = (double*)malloc(sizeof(double) * (size_t)K);
    for (int kk = 0; kk < K; ++kk)
        for (int cc = 0; cc < nc; ++cc)
            S[(size_t)kk * nc + cc] =
                c->h0 ? (double)c->h0[(((size_t)b * H + h) * K + kk) * V + c0 + cc] : 0.0;

    for (int t = 0; t < T; ++t) {
        const size_t row = ((size_t)b * T + t) * H + h;
        if (c->H_in && c->seg_len > 0 && t % c->seg_len == 0) {
            const int s = t / c->seg_len;
            const size_t base = (((size_t)s * c->B + b) * H + h) * (size_t)K * V;
            for (int kk = 0; kk < K; ++kk)
                for (int cc = 0; cc < nc; ++cc)
                    c->H_in[base + (size_t)kk * V + c0 + cc] = S[(size_t)kk * nc + cc];
        }
        const double decay = exp((double)c->g[row]);
        const double bt = (double)c->beta[row];
        for (int kk = 0; kk < K; ++kk) {
            kt[kk] = (double)c->k[row * K + kk];
            qt[kk] = (double)c->q[row * K + kk];
        }
        for (int cc = 0; cc < nc; ++cc) {
            /* k_t @ H_{t-1}, column cc */
            double read = 0.0;
            for (int kk = 0; kk < K; ++kk) read += kt[kk] * S[(size_t)kk * nc + cc];
            if (c->decay_first) read *= decay;   /* k_t @ (exp(g_t) H_{t-1}) */
            const double resid = bt * ((double)c->v[row * V + c0 + cc] - read);
            /* H_t = exp(g_t) H_{t-1} + k_t residual_t^T, then o_t = q_t @ H_t */
            double out = 0.0;
            for (int kk = 0; kk < K; ++kk) {
                double* s = &S[(size_t)kk * nc + cc];
                *s = decay * (*s) + kt[kk] * resid;
                out += qt[kk] * (*s);
            }
            if (c->o) c->o[row * V + c0 + cc] = out;
        }
    }
    if (c->h_final)
        for (int kk = 0; kk < K; ++kk)
            for (int cc = 0; cc < nc; ++cc)
                c->h_final[(((size_t)b * H + h) * K + kk) * V + c0 + cc] = S[(size_t)kk * nc + cc];
    free(S);
    free(kt);
    free(qt);
}

/* seg_len > 0 and H_in != NULL: H_in[s] receives the state entering token s*seg_len.
 * col_block <= 0 means all V columns in one unit.                                       */
void oracle_recurrence(int B, int T, int H, int K, int V, int seg_len, const float* q,
                       const float* k, const float* v, const float* g, const float* beta,
                       const float* h0, double* o, double* h_final, double* H_in,
                       int col_block, int nthreads, int decay_first) {
    rec_ctx c = {B, T, H, K, V, seg_len, col_block > 0 ? col_block : V,
                 q, k, v, g, beta, h0, o, h_final, H_in, decay_first};
    const long nblk = (V + c.col_block - 1) / c.col_block;
    run_units(rec_unit, &c, (long)B * H * nblk, nthreads);
}

/* ------------------------------------------------------------------------------------ */
/* 2. Segment summary ([RFC] 2.2): H_out = M @ H_in + S for one contiguous segment.      */
/* Substituting H_{t-1} = M H_in + S into the recurrence gives the per-token update      */
/*   x = k^T M,  y = k^T S                                                               */
/*   M <- exp(g) M - beta k x^T                                                          */
/*   S <- exp(g) S - beta k y^T + beta k v^T                                             */
/* starting from M = I, S = 0 (rank-1 form; no K^3 products).                            */
/* ------------------------------------------------------------------------------------ */
typedef struct {
    int B, T, H, K, V, nseg;
    const float *k, *v, *g, *beta;
    double *M, *S;
    int decay_first;
} sum_ctx;

static void sum_unit(void* vctx, long unit) {
    const sum_ctx* c = (const sum_ctx*)vctx;
    const int K = c->K, V = c->V, H = c->H, T = c->T;
    const int seg_len = T / c->nseg;
    const int s = (int)(unit % c->nseg);
    const long bh = unit / c->nseg;
    const int b = (int)(bh / H), h = (int)(bh % H);
    double* M = c->M + (((size_t)s * c->B + b) * H + h) * (size_t)K * K;
    double* S = c->S + (((size_t)s * c->B + b) * H + h) * (size_t)K * V;
    double* x = (double*)malloc(sizeof(double) * (size_t)K);
    double* y = (double*)malloc(sizeof(double) * (size_t)V);
    double* kt = (double*)malloc(sizeof(double) * (size_t)K);
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < K; ++j) M[(size_t)i * K + j] = (i == j) ? 1.0 : 0.0;
    for (size_t i = 0; i < (size_t)K * V; ++i) S[i] = 0.0;

    for (int t = s * seg_len; t < (s + 1) * seg_len; ++t) {
        const size_t row = ((size_t)b * T + t) * H + h;
        const double decay = exp((double)c->g[row]);
        const double bt = (double)c->beta[row];
        for (int i = 0; i < K; ++i) kt[i] = (double)c->k[row * K + i];
        for (int j = 0; j < K; ++j) {
            double a = 0.0;
            for (int i = 0; i < K; ++i) a += kt[i] * M[(size_t)i * K + j];
            x[j] = a;
        }
        for (int j = 0; j < V; ++j) {
            double a = 0.0;
            for (int i = 0; i < K; ++i) a += kt[i] * S[(size_t)i * V + j];
            y[j] = a;
        }
        for (int i = 0; i < K; ++i) {
            const double bk = bt * kt[i];
            /* the read's correction is decayed too when the decayed state is read */
            const double rk = c->decay_first ? decay * bk : bk;
            for (int j = 0; j < K; ++j) M[(size_t)i * K + j] = decay * M[(size_t)i * K + j] - rk * x[j];
            for (int j = 0; j < V; ++j)
                S[(size_t)i * V + j] =
                    decay * S[(size_t)i * V + j] - rk * y[j] + bk * (double)c->v[row * V + j];
        }
    }
    free(x);
    free(y);
    free(kt);
}

void oracle_summary(int B, int T, int H, int K, int V, int nseg, const float* k, const float* v,
                    const float* g, const float* beta, double* M, double* S, int nthreads,
                    int decay_first) {
    sum_ctx c = {B, T, H, K, V, nseg, k, v, g, beta, M, S, decay_first};
    run_units(sum_unit, &c, (long)B * H * nseg, nthreads);
}

/* ------------------------------------------------------------------------------------ */
/* 3. Compose ([RFC] 2.2; [ART] "Then parallelize across GPUs"): segment 0 then          */
/* segment 1 is  M = M1 @ M0,  S = M1 @ S0 + S1.  One (b,h) pair.                         */
/* ------------------------------------------------------------------------------------ */
void oracle_compose(int K, int V, const double* M1, const double* S1, const double* M0,
                    const double* S0, double* M, double* S) {
    for (int i = 0; i < K; ++i) {
        for (int j = 0; j < K; ++j) {
            double a = 0.0;
            for (int l = 0; l < K; ++l) a += M1[(size_t)i * K + l] * M0[(size_t)l * K + j];
            M[(size_t)i * K + j] = a;
        }
        for (int j = 0; j < V; ++j) {
            double a = S1[(size_t)i * V + j];
            for (int l = 0; l < K; ++l) a += M1[(size_t)i * K + l] * S0[(size_t)l * V + j];
            S[(size_t)i * V + j] = a;
        }
    }
}

/* ------------------------------------------------------------------------------------ */
/* 4. Exclusive in-order scan of segment summaries: H_in[0] = h0 (zero when NULL),        */
/* H_in[s] = M[s-1] @ H_in[s-1] + S[s-1]. "Every segment starts from the previous         */
/* segment's final state" ([RFC] 2.1 last paragraph; [ART] prefix scan, made exclusive). */
/* BH = B*H heads; M [nseg,BH,K,K], S/H_in [nseg,BH,K,V], h0 [BH,K,V].                    */
/* ------------------------------------------------------------------------------------ */
void oracle_scan(int nseg, int BH, int K, int V, const double* M, const double* S,
                 const double* h0, double* H_in) {
    const size_t kk = (size_t)K * K, kv = (size_t)K * V;
    for (int bh = 0; bh < BH; ++bh) {
        double* first = H_in + (size_t)bh * kv;
        for (size_t i = 0; i < kv; ++i) first[i] = h0 ? h0[(size_t)bh * kv + i] : 0.0;
        for (int s = 1; s < nseg; ++s) {
            const double* Mp = M + ((size_t)(s - 1) * BH + bh) * kk;
            const double* Sp = S + ((size_t)(s - 1) * BH + bh) * kv;
            const double* Hp = H_in + ((size_t)(s - 1) * BH + bh) * kv;
            double* Hn = H_in + ((size_t)s * BH + bh) * kv;
            for (int i = 0; i < K; ++i)
                for (int j = 0; j < V; ++j) {
                    double a = Sp[(size_t)i * V + j];
                    for (int l = 0; l < K; ++l) a += Mp[(size_t)i * K + l] * Hp[(size_t)l * V + j];
                    Hn[(size_t)i * V + j] = a;
                }
        }
    }
}

/* ------------------------------------------------------------------------------------ */
/* 5. Chunked form ([ART] 08, "First parallelize within a GPU"), restated for the         */
/* un-decayed read of [RFC] 2.1. Within one chunk of c tokens, with G_i the inclusive    */
/* cumulative sum of g inside the chunk and Gx_i = G_i - g_i the exclusive one:          */
/*   P[i,j] = exp(Gx_i - G_j) (k_i . k_j)  for j < i         (decay-weighted key Gram)    */
/*   A      = (I + diag(beta) P)^{-1}                         (unit lower triangular)     */
/*   U      = A diag(beta) V,   W = A diag(beta) Kr,   Kr_i = exp(Gx_i) k_i              */
/*   R      = U - W H_start                                  (corrected values)           */
/*   C[i,j] = exp(G_i - G_j) (q_i . k_j)  for j <= i                                     */
/*   O      = Qd H_start + C R,   Qd_i = exp(G_i) q_i                                     */
/*   H_end  = exp(G_last) H_start + Kd^T R,   Kd_j = exp(G_last - G_j) k_j               */
/* and the chunk's own summary  M_n = exp(G_last) I - Kd^T W,  E_n = Kd^T U.              */
/* This exists to pin "chunked == per-token" and to expose chunk intermediates.         */
/* ------------------------------------------------------------------------------------ */
typedef struct {
    int B, T, H, K, V, chunk, nseg;
    const float *q, *k, *v, *g, *beta, *h0;
    double *o, *h_final, *M, *S;
    int decay_first;   /* the read sees exp(g_i) times the state: G_i in P and Kr, not Gx_i */
} chk_ctx;

/* forward substitution for A = (I + L)^{-1}, L strictly lower (n x n, row-major) */
static void unit_lower_inverse(int n, const double* L, double* A) {
    for (int j = 0; j < n; ++j) {
        for (int i = 0; i < n; ++i) A[(size_t)i * n + j] = 0.0;
        A[(size_t)j * n + j] = 1.0;
        for (int i = j + 1; i < n; ++i) {
            double a = 0.0;
            for (int l = j; l < i; ++l) a += L[(size_t)i * n + l] * A[(size_t)l * n + j];
            A[(size_t)i * n + j] = -a;
        }
    }
}

/* One chunk: reads Hs (K x V), writes O rows (if o != NULL), overwrites Hs with H_end.
 * If Mn/En are non-NULL, also writes the chunk summary.                                 */
static void chunk_step(const chk_ctx* c, int b, int h, int t0, int n, double* Hs, double* Mn,
                       double* En, double* work) {
    const int K = c->K, V = c->V, H = c->H;
    double* G = work;                     /* n   */
    double* Gx = G + n;                   /* n   */
    double* bt = Gx + n;                  /* n   */
    double* kd = bt + n;                  /* n*K */
    double* qd = kd + (size_t)n * K;      /* n*K */
    double* vd = qd + (size_t)n * K;      /* n*V */
    double* L = vd + (size_t)n * V;       /* n*n */
    double* A = L + (size_t)n * n;        /* n*n */
    double* Cm = A + (size_t)n * n;       /* n*n */
    double* U = Cm + (size_t)n * n;       /* n*V */
    double* W = U + (size_t)n * V;        /* n*K */
    double* R = W + (size_t)n * K;        /* n*V */
    double acc = 0.0;
    for (int i = 0; i < n; ++i) {
        const size_t row = ((size_t)b * c->T + t0 + i) * H + h;
        const double gi = (double)c->g[row];
        Gx[i] = acc;
        acc += gi;
        G[i] = acc;
        bt[i] = (double)c->beta[row];
        for (int j = 0; j < K; ++j) {
            kd[(size_t)i * K + j] = (double)c->k[row * K + j];
            qd[(size_t)i * K + j] = c->q ? (double)c->q[row * K + j] : 0.0;
        }
        for (int j = 0; j < V; ++j) vd[(size_t)i * V + j] = (double)c->v[row * V + j];
    }
    const double Glast = G[n - 1];
    const double* Gr = c->decay_first ? G : Gx;   /* cumulative gate of the read side */
    /* L = diag(beta) P */
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < n; ++j) {
            double p = 0.0, cq = 0.0;
            if (j < i) {
                double d = 0.0;
                for (int l = 0; l < K; ++l) d += kd[(size_t)i * K + l] * kd[(size_t)j * K + l];
                p = exp(Gr[i] - G[j]) * d;
            }
            if (j <= i) {
                double d = 0.0;
                for (int l = 0; l < K; ++l) d += qd[(size_t)i * K + l] * kd[(size_t)j * K + l];
                cq = exp(G[i] - G[j]) * d;
            }
            L[(size_t)i * n + j] = bt[i] * p;
            Cm[(size_t)i * n + j] = cq;
        }
    unit_lower_inverse(n, L, A);
    /* U = A diag(beta) V ; W = A diag(beta) Kr */
    for (int i = 0; i < n; ++i) {
        for (int j = 0; j < V; ++j) {
            double a = 0.0;
            for (int l = 0; l <= i; ++l) a += A[(size_t)i * n + l] * bt[l] * vd[(size_t)l * V + j];
            U[(size_t)i * V + j] = a;
        }
        for (int j = 0; j < K; ++j) {
            double a = 0.0;
            for (int l = 0; l <= i; ++l)
                a += A[(size_t)i * n + l] * bt[l] * exp(Gr[l]) * kd[(size_t)l * K + j];
            W[(size_t)i * K + j] = a;
        }
    }
    /* R = U - W Hs */
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < V; ++j) {
            double a = U[(size_t)i * V + j];
            for (int l = 0; l < K; ++l) a -= W[(size_t)i * K + l] * Hs[(size_t)l * V + j];
            R[(size_t)i * V + j] = a;
        }
    /* O = Qd Hs + C R */
    if (c->o) {
        for (int i = 0; i < n; ++i) {
            const size_t row = ((size_t)b * c->T + t0 + i) * H + h;
            for (int j = 0; j < V; ++j) {
                double a = 0.0;
                for (int l = 0; l < K; ++l) a += qd[(size_t)i * K + l] * Hs[(size_t)l * V + j];
                a *= exp(G[i]);
                for (int l = 0; l <= i; ++l) a += Cm[(size_t)i * n + l] * R[(size_t)l * V + j];
                c->o[row * V + j] = a;
            }
        }
    }
    /* chunk summary, M_n = exp(G_last) I - Kd^T W, E_n = Kd^T U */
    if (Mn && En) {
        for (int r = 0; r < K; ++r) {
            for (int j = 0; j < K; ++j) {
                double a = (r == j) ? exp(Glast) : 0.0;
                for (int l = 0; l < n; ++l)
                    a -= exp(Glast - G[l]) * kd[(size_t)l * K + r] * W[(size_t)l * K + j];
                Mn[(size_t)r * K + j] = a;
            }
            for (int j = 0; j < V; ++j) {
                double a = 0.0;
                for (int l = 0; l < n; ++l)
                    a += exp(Glast - G[l]) * kd[(size_t)l * K + r] * U[(size_t)l * V + j];
                En[(size_t)r * V + j] = a;
            }
        }
    }
    /* H_end = exp(G_last) Hs + Kd^T R */
    for (int r = 0; r < K; ++r)
        for (int j = 0; j < V; ++j) {
            double a = exp(Glast) * Hs[(size_t)r * V + j];
            for (int l = 0; l < n; ++l)
                a += exp(Glast - G[l]) * kd[(size_t)l * K + r] * R[(size_t)l * V + j];
            Hs[(size_t)r * V + j] = a;
        }
}

static size_t chunk_work_doubles(int n, int K, int V) {
    return (size_t)3 * n + (size_t)n * K * 3 + (size_t)n * V * 3 + (size_t)n * n * 3;
}

static void chk_fwd_unit(void* vctx, long unit) {
    const chk_ctx* c = (const chk_ctx*)vctx;
    const int K = c->K, V = c->V, H = c->H;
    const int b = (int)(unit / H), h = (int)(unit % H);
    double* Hs = (double*)malloc(sizeof(double) * (size_t)K * V);
    double* work = (double*)malloc(sizeof(double) * chunk_work_doubles(c->chunk, K, V));
    for (int kk = 0; kk < K; ++kk)
        for (int j = 0; j < V; ++j)
            Hs[(size_t)kk * V + j] = c->h0 ? (double)c->h0[(((size_t)b * H + h) * K + kk) * V + j] : 0.0;
    for (int t0 = 0; t0 < c->T; t0 += c->chunk) {
        const int n = (t0 + c->chunk <= c->T) ? c->chunk : c->T - t0;
        chunk_step(c, b, h, t0, n, Hs, NULL, NULL, work);
    }
    if (c->h_final)
        for (size_t i = 0; i < (size_t)K * V; ++i)
            c->h_final[((size_t)b * H + h) * (size_t)K * V + i] = Hs[i];
    free(Hs);
    free(work);
}

/* Chunked forward from h0 over all T tokens (the last chunk may be short). */
void oracle_chunked_fwd(int B, int T, int H, int K, int V, int chunk, const float* q, const float* k,
                        const float* v, const float* g, const float* beta, const float* h0,
                        double* o, double* h_final, int nthreads, int decay_first) {
    chk_ctx c = {B, T, H, K, V, chunk, 1, q, k, v, g, beta, h0, o, h_final, NULL, NULL, decay_first};
    run_units(chk_fwd_unit, &c, (long)B * H, nthreads);
}

static void chk_sum_unit(void* vctx, long unit) {
    const chk_ctx* c = (const chk_ctx*)vctx;
    const int K = c->K, V = c->V, H = c->H;
    const int seg_len = c->T / c->nseg;
    const int s = (int)(unit % c->nseg);
    const long bh = unit / c->nseg;
    const int b = (int)(bh / H), h = (int)(bh % H);
    double* Mseg = c->M + (((size_t)s * c->B + b) * H + h) * (size_t)K * K;
    double* Sseg = c->S + (((size_t)s * c->B + b) * H + h) * (size_t)K * V;
    double* Mn = (double*)malloc(sizeof(double) * (size_t)K * K);
    double* En = (double*)malloc(sizeof(double) * (size_t)K * V);
    double* Mt = (double*)malloc(sizeof(double) * (size_t)K * K);
    double* St = (double*)malloc(sizeof(double) * (size_t)K * V);
    double* Hs = (double*)malloc(sizeof(double) * (size_t)K * V);
    double* work = (double*)malloc(sizeof(double) * chunk_work_doubles(c->chunk, K, V));
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < K; ++j) Mseg[(size_t)i * K + j] = (i == j) ? 1.0 : 0.0;
    for (size_t i = 0; i < (size_t)K * V; ++i) Sseg[i] = 0.0;
    for (int t0 = s * seg_len; t0 < (s + 1) * seg_len; t0 += c->chunk) {
        const int n = (t0 + c->chunk <= (s + 1) * seg_len) ? c->chunk : (s + 1) * seg_len - t0;
        for (size_t i = 0; i < (size_t)K * V; ++i) Hs[i] = 0.0;
        chunk_step(c, b, h, t0, n, Hs, Mn, En, work);
        /* segment-so-far (Mseg, Sseg) then this chunk (Mn, En) */
        oracle_compose(K, V, Mn, En, Mseg, Sseg, Mt, St);
        memcpy(Mseg, Mt, sizeof(double) * (size_t)K * K);
        memcpy(Sseg, St, sizeof(double) * (size_t)K * V);
    }
    free(Mn);
    free(En);
    free(Mt);
    free(St);
    free(Hs);
    free(work);
}

/* Per-segment summaries built from the chunk summaries (M_n, E_n) composed in order. */
void oracle_chunked_summary(int B, int T, int H, int K, int V, int chunk, int nseg, const float* k,
                            const float* v, const float* g, const float* beta, double* M,
                            double* S, int nthreads, int decay_first) {
    chk_ctx c = {B, T, H, K, V, chunk, nseg, NULL, k, v, g, beta, NULL, NULL, NULL, M, S, decay_first};
    run_units(chk_sum_unit, &c, (long)B * H * nseg, nthreads);
}

/* ------------------------------------------------------------------------------------ */
/* 5. Per-channel gates ([KDA] "KDA Chunk Backward -- TPU/Pallas Kernel Design", section */
/* 1.2: the state decays row by row, 2^(g) with g in R^K per token). With a = exp(g_t)   */
/* per key channel, one token does                                                        */
/*   read before the decay:  r = beta (v - H^T k),    H <- diag(a) H + k r^T             */
/*   decayed read (flag):    H' = diag(a) H, r = beta (v - H'^T k),  H <- H' + k r^T    */
/* and o_t = H_t^T q_t. Written on its own, not through the scalar-gate code above: with */
/* equal channels it must reproduce that code (a pin), so it may not share it.            */
/* Gate layout: g [B, T, H, K].                                                           */
/* ------------------------------------------------------------------------------------ */
typedef struct {
    int B, T, H, K, V, seg_len, col_block;
    const float *q, *k, *v, *g, *beta, *h0;
    double *o, *h_final, *H_in;
    int decay_first;
} kda_ctx;

static void kda_rec_unit(void* vctx, long unit) {
    const kda_ctx* c = (const kda_ctx*)vctx;
    const int K = c->K, V = c->V, H = c->H, T = c->T, cb = c->col_block;
    const long nblk = (V + cb - 1) / cb;
    const int blk = (int)(unit % nblk);
    const long bh = unit / nblk;
    const int b = (int)(bh / H), h = (int)(bh % H);
    const int v0 = blk * cb, v1 = (v0 + cb < V) ? v0 + cb : V, w = v1 - v0;
    double* St = (double*)malloc(sizeof(double) * (size_t)K * w);   /* state columns v0..v1 */
    double* r = (double*)malloc(sizeof(double) * (size_t)w);
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < w; ++j)
            St[(size_t)i * w + j] =
                c->h0 ? (double)c->h0[(((size_t)b * H + h) * K + i) * V + v0 + j] : 0.0;
    for (int t = 0; t < T; ++t) {
        if (c->H_in && c->seg_len > 0 && t % c->seg_len == 0) {
            const int s = t / c->seg_len;
            for (int i = 0; i < K; ++i)
                for (int j = 0; j < w; ++j)
                    c->H_in[((((size_t)s * c->B + b) * H + h) * K + i) * V + v0 + j] =
                        St[(size_t)i * w + j];
        }
        const size_t row = ((size_t)b * T + t) * H + h;
        const float* kt = c->k + row * K;
        const float* gt = c->g + row * K;
        const double bt = (double)c->beta[row];
        if (c->decay_first)   /* decay every row of the state before the read */
            for (int i = 0; i < K; ++i) {
                const double a = exp((double)gt[i]);
                for (int j = 0; j < w; ++j) St[(size_t)i * w + j] *= a;
            }
        for (int j = 0; j < w; ++j) {   /* r = beta (v - H^T k) */
            double acc = 0.0;
            for (int i = 0; i < K; ++i) acc += (double)kt[i] * St[(size_t)i * w + j];
            r[j] = bt * ((double)c->v[row * V + v0 + j] - acc);
        }
        for (int i = 0; i < K; ++i) {
            const double a = c->decay_first ? 1.0 : exp((double)gt[i]);
            for (int j = 0; j < w; ++j)
                St[(size_t)i * w + j] = a * St[(size_t)i * w + j] + (double)kt[i] * r[j];
        }
        if (c->o)
            for (int j = 0; j < w; ++j) {
                double acc = 0.0;
                for (int i = 0; i < K; ++i) acc += (double)c->q[row * K + i] * St[(size_t)i * w + j];
                c->o[row * V + v0 + j] = acc;
            }
    }
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < w; ++j)
            c->h_final[(((size_t)b * H + h) * K + i) * V + v0 + j] = St[(size_t)i * w + j];
    free(St);
    free(r);
}

void oracle_kda_recurrence(int B, int T, int H, int K, int V, int seg_len, const float* q,
                           const float* k, const float* v, const float* g, const float* beta,
                           const float* h0, double* o, double* h_final, double* H_in,
                           int col_block, int nthreads, int decay_first) {
    kda_ctx c = {B, T, H, K, V, seg_len, col_block > 0 ? col_block : V,
                 q, k, v, g, beta, h0, o, h_final, H_in, decay_first};
    const long nblk = (V + c.col_block - 1) / c.col_block;
    run_units(kda_rec_unit, &c, (long)B * H * nblk, nthreads);
}

/* Per-segment summaries with per-channel gates: H_out = M H_in + S over a segment. One   */
/* token maps H to T_t H + beta k v^T with T_t = diag(a) - beta k k^T (read before the    */
/* decay) or (I - beta k k^T) diag(a) (decayed read); M is the product of the T_t from I, */
/* S the state reached from 0.                                                             */
typedef struct {
    int B, T, H, K, V, nseg;
    const float *k, *v, *g, *beta;
    double *M, *S;
    int decay_first;
} kda_sum_ctx;

/* X (K x n) <- T_t X + beta k u^T for one token, u = v (S) or 0 (M) */
static void kda_apply(int K, int n, double* X, const double* a, const double* kt, double bt,
                      const float* vrow, int decay_first, double* y) {
    if (decay_first)
        for (int i = 0; i < K; ++i)
            for (int j = 0; j < n; ++j) X[(size_t)i * n + j] *= a[i];
    for (int j = 0; j < n; ++j) {   /* y = k^T X (X already decayed when the read is) */
        double acc = 0.0;
        for (int i = 0; i < K; ++i) acc += kt[i] * X[(size_t)i * n + j];
        y[j] = acc;
    }
    for (int i = 0; i < K; ++i) {
        const double ai = decay_first ? 1.0 : a[i];
        for (int j = 0; j < n; ++j)
            X[(size_t)i * n + j] = ai * X[(size_t)i * n + j] - bt * kt[i] * y[j] +
                                   (vrow ? bt * kt[i] * (double)vrow[j] : 0.0);
    }
}

static void kda_sum_unit(void* vctx, long unit) {
    const kda_sum_ctx* c = (const kda_sum_ctx*)vctx;
    const int K = c->K, V = c->V, H = c->H, T = c->T;
    const int seg_len = T / c->nseg;
    const int s = (int)(unit % c->nseg);
    const long bh = unit / c->nseg;
    const int b = (int)(bh / H), h = (int)(bh % H);
    double* M = c->M + (((size_t)s * c->B + b) * H + h) * (size_t)K * K;
    double* S = c->S + (((size_t)s * c->B + b) * H + h) * (size_t)K * V;
    double* a = (double*)malloc(sizeof(double) * (size_t)K);
    double* kt = (double*)malloc(sizeof(double) * (size_t)K);
    double* y = (double*)malloc(sizeof(double) * (size_t)(K > V ? K : V));
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < K; ++j) M[(size_t)i * K + j] = (i == j) ? 1.0 : 0.0;
    for (size_t i = 0; i < (size_t)K * V; ++i) S[i] = 0.0;
    for (int t = s * seg_len; t < (s + 1) * seg_len; ++t) {
        const size_t row = ((size_t)b * T + t) * H + h;
        for (int i = 0; i < K; ++i) {
            a[i] = exp((double)c->g[row * K + i]);
            kt[i] = (double)c->k[row * K + i];
        }
        const double bt = (double)c->beta[row];
        kda_apply(K, K, M, a, kt, bt, NULL, c->decay_first, y);
        kda_apply(K, V, S, a, kt, bt, c->v + row * V, c->decay_first, y);
    }
    free(a);
    free(kt);
    free(y);
}

void oracle_kda_summary(int B, int T, int H, int K, int V, int nseg, const float* k,
                        const float* v, const float* g, const float* beta, double* M, double* S,
                        int nthreads, int decay_first) {
    kda_sum_ctx c = {B, T, H, K, V, nseg, k, v, g, beta, M, S, decay_first};
    run_units(kda_sum_unit, &c, (long)B * H * nseg, nthreads);
}

/* ------------------------------------------------------------------------------------ */
/* 6. Backward of the per-token recurrence ([RFC] 6.4.3, the reverse flow that ends in   */
/* dQ, dK, dV, dg, dbeta; [KDA] "KDA Chunk Backward -- TPU/Pallas Kernel Design" 1, the  */
/* gradients it produces, dh0 included). The loss is                                      */
/*   L = sum_t do_t . o_t + <dht, h_final>                                                */
/* With P = H_{t-1}, a = exp(g_t), c = 1 (or a for the decayed read), one token is        */
/*   x = P^T k,  r = beta (v - c x),  H_t = a P + k r^T,  o = H_t^T q.                    */
/* Walking the tokens backwards with D = dL/dH_t from the later tokens:                   */
/*   G  = D + q do^T                  dq = H_t do                                         */
/*   dr = G^T k                       dk = G r + c P dx',  dx' = -beta dr                  */
/*   dv = beta dr                     dbeta = dr . (v - c x)                              */
/*   da = <G, P> (+ dx' . x when c = a)                 dg = a da                         */
/*   D  <- a G + c k dx'^T            (the gradient on H_{t-1})                            */
/* and dh0 is D after token 0. The states H_{t-1} are recomputed block by block from      */
/* checkpoints taken every ~sqrt(T) tokens of a first forward walk. One unit = one head.  */
/* ------------------------------------------------------------------------------------ */
typedef struct {
    int B, T, H, K, V;
    const float *q, *k, *v, *g, *beta, *h0, *dO, *dht;
    double *dq, *dk, *dv, *dg, *dbeta, *dh0;
    int decay_first;
} bwd_ctx;

/* one forward token on a K x V state X (in place) */
static void fwd_token(int K, int V, double* X, const float* kt, const float* vt, double a,
                      double bt, int decay_first, double* x) {
    const double cr = decay_first ? a : 1.0;
    for (int j = 0; j < V; ++j) {
        double acc = 0.0;
        for (int i = 0; i < K; ++i) acc += (double)kt[i] * X[(size_t)i * V + j];
        x[j] = bt * ((double)vt[j] - cr * acc);   /* the residual r */
    }
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < V; ++j)
            X[(size_t)i * V + j] = a * X[(size_t)i * V + j] + (double)kt[i] * x[j];
}

static void bwd_unit(void* vctx, long unit) {
    const bwd_ctx* c = (const bwd_ctx*)vctx;
    const int K = c->K, V = c->V, H = c->H, T = c->T;
    const int b = (int)(unit / H), h = (int)(unit % H);
    const size_t KV = (size_t)K * V;
    int blk = 1;
    while (blk * blk < T) ++blk;
    const int nblk = (T + blk - 1) / blk;
    double* ck = (double*)malloc(sizeof(double) * KV * (size_t)nblk);      /* state entering block */
    double* st = (double*)malloc(sizeof(double) * KV * (size_t)(blk + 1)); /* states inside a block */
    double* D = (double*)malloc(sizeof(double) * KV);
    double* G = (double*)malloc(sizeof(double) * KV);
    double* x = (double*)malloc(sizeof(double) * (size_t)V);
    double* r = (double*)malloc(sizeof(double) * (size_t)V);
    double* dr = (double*)malloc(sizeof(double) * (size_t)V);
    double* dxp = (double*)malloc(sizeof(double) * (size_t)V);
    const size_t head = ((size_t)b * H + h) * KV;

    /* forward walk: checkpoints */
    for (size_t e = 0; e < KV; ++e) st[e] = c->h0 ? (double)c->h0[head + e] : 0.0;
    for (int t = 0; t < T; ++t) {
        if (t % blk == 0) memcpy(ck + (size_t)(t / blk) * KV, st, sizeof(double) * KV);
        const size_t row = ((size_t)b * T + t) * H + h;
        fwd_token(K, V, st, c->k + row * K, c->v + row * V, exp((double)c->g[row]),
                  (double)c->beta[row], c->decay_first, x);
    }
    for (size_t e = 0; e < KV; ++e) D[e] = c->dht ? (double)c->dht[head + e] : 0.0;

    for (int bi = nblk - 1; bi >= 0; --bi) {
        const int t0 = bi * blk, n = (t0 + blk <= T) ? blk : T - t0;
        memcpy(st, ck + (size_t)bi * KV, sizeof(double) * KV);
        for (int i = 0; i < n; ++i) {
            memcpy(st + (size_t)(i + 1) * KV, st + (size_t)i * KV, sizeof(double) * KV);
            const size_t row = ((size_t)b * T + t0 + i) * H + h;
            fwd_token(K, V, st + (size_t)(i + 1) * KV, c->k + row * K, c->v + row * V,
                      exp((double)c->g[row]), (double)c->beta[row], c->decay_first, x);
        }
        for (int i = n - 1; i >= 0; --i) {
            const int t = t0 + i;
            const size_t row = ((size_t)b * T + t) * H + h;
            const double* P = st + (size_t)i * KV;
            const double* Ht = st + (size_t)(i + 1) * KV;
            const float *qt = c->q + row * K, *kt = c->k + row * K, *vt = c->v + row * V;
            const float* dot = c->dO + row * V;
            const double a = exp((double)c->g[row]), bt = (double)c->beta[row];
            const double cr = c->decay_first ? a : 1.0;
            for (int kk = 0; kk < K; ++kk)
                for (int j = 0; j < V; ++j)
                    G[(size_t)kk * V + j] = D[(size_t)kk * V + j] + (double)qt[kk] * (double)dot[j];
            for (int kk = 0; kk < K; ++kk) {   /* dq = H_t do */
                double acc = 0.0;
                for (int j = 0; j < V; ++j) acc += Ht[(size_t)kk * V + j] * (double)dot[j];
                c->dq[row * K + kk] = acc;
            }
            double dbeta = 0.0;
            for (int j = 0; j < V; ++j) {
                double xa = 0.0, da_ = 0.0;
                for (int kk = 0; kk < K; ++kk) {
                    xa += (double)kt[kk] * P[(size_t)kk * V + j];
                    da_ += G[(size_t)kk * V + j] * (double)kt[kk];
                }
                x[j] = xa;
                r[j] = bt * ((double)vt[j] - cr * xa);
                dr[j] = da_;
                c->dv[row * V + j] = bt * da_;
                dbeta += da_ * ((double)vt[j] - cr * xa);
                dxp[j] = -bt * da_;
            }
            c->dbeta[row] = dbeta;
            double da = 0.0;
            for (size_t e = 0; e < KV; ++e) da += G[e] * P[e];
            if (c->decay_first)
                for (int j = 0; j < V; ++j) da += dxp[j] * x[j];
            for (int kk = 0; kk < K; ++kk) {
                double acc = 0.0;
                for (int j = 0; j < V; ++j)
                    acc += G[(size_t)kk * V + j] * r[j] + cr * P[(size_t)kk * V + j] * dxp[j];
                c->dk[row * K + kk] = acc;
            }
            c->dg[row] = a * da;
            for (int kk = 0; kk < K; ++kk)
                for (int j = 0; j < V; ++j)
                    D[(size_t)kk * V + j] = a * G[(size_t)kk * V + j] + cr * (double)kt[kk] * dxp[j];
        }
    }
    if (c->dh0) memcpy(c->dh0 + head, D, sizeof(double) * KV);
    free(ck); free(st); free(D); free(G); free(x); free(r); free(dr); free(dxp);
}

void oracle_backward(int B, int T, int H, int K, int V, const float* q, const float* k,
                     const float* v, const float* g, const float* beta, const float* h0,
                     const float* dO, const float* dht, double* dq, double* dk, double* dv,
                     double* dg, double* dbeta, double* dh0, int nthreads, int decay_first) {
    bwd_ctx c = {B, T, H, K, V, q, k, v, g, beta, h0, dO, dht,
                 dq, dk, dv, dg, dbeta, dh0, decay_first};
    run_units(bwd_unit, &c, (long)B * H, nthreads);
}

/* ------------------------------------------------------------------------------------ */
/* 7. State-gradient summary of one segment ([RFC] 6.4.3: the summary step yields         */
/* dS_local, the gradient reaching the state that enters the segment from the segment's  */
/* own outputs). The gradient on the state obeys the transposed token transition; the     */
/* transition exp(g) I - beta k k^T (or exp(g) (I - beta k k^T)) is symmetric, so one     */
/* token backwards is, in rank-1 form,                                                    */
/*   G = D + q do^T,   y = k^T G,   D <- exp(g) G - c beta k y^T   (c as in section 6)    */
/* started at the segment's last token from dH_end[s] (zero when dH_end is NULL) and read */
/* out after its first token. Needs neither v nor any forward state. One unit = one       */
/* (b, h, segment). dS and dH_end are [nseg, B, H, K, V].                                 */
/* ------------------------------------------------------------------------------------ */
typedef struct {
    int B, T, H, K, V, nseg;
    const float *q, *k, *g, *beta, *dO;
    const double* dH_end;
    double* dS;
    int decay_first;
} sgs_ctx;

static void sgs_unit(void* vctx, long unit) {
    const sgs_ctx* c = (const sgs_ctx*)vctx;
    const int K = c->K, V = c->V, H = c->H, T = c->T;
    const int seg_len = T / c->nseg;
    const int s = (int)(unit % c->nseg);
    const long bh = unit / c->nseg;
    const int b = (int)(bh / H), h = (int)(bh % H);
    const size_t KV = (size_t)K * V;
    double* D = c->dS + (((size_t)s * c->B + b) * H + h) * KV;
    double* y = (double*)malloc(sizeof(double) * (size_t)V);
    for (size_t e = 0; e < KV; ++e)
        D[e] = c->dH_end ? c->dH_end[(((size_t)s * c->B + b) * H + h) * KV + e] : 0.0;
    for (int t = (s + 1) * seg_len - 1; t >= s * seg_len; --t) {
        const size_t row = ((size_t)b * T + t) * H + h;
        const float *qt = c->q + row * K, *kt = c->k + row * K, *dot = c->dO + row * V;
        const double a = exp((double)c->g[row]), bt = (double)c->beta[row];
        const double cr = c->decay_first ? a : 1.0;
        for (int i = 0; i < K; ++i)
            for (int j = 0; j < V; ++j) D[(size_t)i * V + j] += (double)qt[i] * (double)dot[j];
        for (int j = 0; j < V; ++j) {
            double acc = 0.0;
            for (int i = 0; i < K; ++i) acc += (double)kt[i] * D[(size_t)i * V + j];
            y[j] = acc;
        }
        for (int i = 0; i < K; ++i)
            for (int j = 0; j < V; ++j)
                D[(size_t)i * V + j] = a * D[(size_t)i * V + j] - cr * bt * (double)kt[i] * y[j];
    }
    free(y);
}

void oracle_state_grad_summary(int B, int T, int H, int K, int V, int nseg, const float* q,
                               const float* k, const float* g, const float* beta,
                               const float* dO, const double* dH_end, double* dS, int nthreads,
                               int decay_first) {
    sgs_ctx c = {B, T, H, K, V, nseg, q, k, g, beta, dO, dH_end, dS, decay_first};
    run_units(sgs_unit, &c, (long)B * H * nseg, nthreads);
}

/* ------------------------------------------------------------------------------------ */
/* 8. Reverse scan of the state gradients ([RFC] 6.4.3, "dH_in = M^T dH_out + dS_local"): */
/* the state after the last segment carries dht (zero when NULL); going back over the     */
/* segments, dH_in[s] = M[s]^T dH_in[s+1] + dS[s] with dH_in[nseg] = dht. dh0 is          */
/* dH_in[0]. M [nseg,BH,K,K], dS / dH_in [nseg,BH,K,V], dht [BH,K,V].                       */
/* ------------------------------------------------------------------------------------ */
void oracle_state_grad_scan(int nseg, int BH, int K, int V, const double* M, const double* dS,
                            const double* dht, double* dH_in) {
    const size_t KV = (size_t)K * V, KK = (size_t)K * K;
    double* cur = (double*)malloc(sizeof(double) * KV);
    for (int bh = 0; bh < BH; ++bh) {
        for (size_t e = 0; e < KV; ++e) cur[e] = dht ? dht[(size_t)bh * KV + e] : 0.0;
        for (int s = nseg - 1; s >= 0; --s) {
            const double* Ms = M + ((size_t)s * BH + bh) * KK;
            double* out = dH_in + ((size_t)s * BH + bh) * KV;
            for (int i = 0; i < K; ++i)
                for (int j = 0; j < V; ++j) {
                    double acc = dS[((size_t)s * BH + bh) * KV + (size_t)i * V + j];
                    for (int m = 0; m < K; ++m) acc += Ms[(size_t)m * K + i] * cur[(size_t)m * V + j];
                    out[(size_t)i * V + j] = acc;
                }
            memcpy(cur, out, sizeof(double) * KV);
        }
    }
    free(cur);
}
