/*
 * synth.c -- seeded synthetic inputs for the gated delta rule (host code, no GPU).
 *
 * This module only draws random numbers and shapes them into inputs; it holds none of the
 * recurrence's arithmetic. Both the CUDA path's harness and the fp64 oracle's tests take
 * their inputs from here, so the two sides see bit-identical values.
 *
 * Generator: xoshiro256** (Blackman & Vigna, 2018), seeded through splitmix64, with one
 * independent stream per row (a row = one (b, t) token with all its heads), so the
 * result does not depend on the number of threads. Normals come from the Box-Muller
 * transform, both outputs used. Values are computed in double and rounded once to the
 * storage type (fp32, or bf16 with round-to-nearest-even, returned as exact floats).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

static uint64_t splitmix64(uint64_t* x) {
    uint64_t z = (*x += 0x9E3779B97F4A7C15ULL);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

typedef struct { uint64_t s[4]; int have_spare; double spare; } rng_t;

static uint64_t rotl(uint64_t x, int k) { return (x << k) | (x >> (64 - k)); }

static uint64_t xoshiro_next(rng_t* r) {
    const uint64_t result = rotl(r->s[1] * 5, 7) * 9;
    const uint64_t t = r->s[1] << 17;
    r->s[2] ^= r->s[0];
    r->s[3] ^= r->s[1];
    r->s[1] ^= r->s[2];
    r->s[0] ^= r->s[3];
    r->s[2] ^= t;
    r->s[3] = rotl(r->s[3], 45);
    return result;
}

static void rng_seed(rng_t* r, uint64_t seed, uint32_t tensor_id, uint64_t row) {
    uint64_t x = seed;
    uint64_t a = splitmix64(&x);
    x = a ^ ((uint64_t)tensor_id * 0xD1B54A32D192ED03ULL);
    uint64_t b = splitmix64(&x);
    x = b ^ (row * 0xABC98388FB8FAC03ULL);
    for (int i = 0; i < 4; ++i) r->s[i] = splitmix64(&x);
    r->have_spare = 0;
    r->spare = 0.0;
}

/* uniform in the open interval (0, 1) */
static double rng_uniform(rng_t* r) {
    return ((double)(xoshiro_next(r) >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static double rng_normal(rng_t* r) {
    if (r->have_spare) {
        r->have_spare = 0;
        return r->spare;
    }
    const double u1 = rng_uniform(r), u2 = rng_uniform(r);
    const double rad = sqrt(-2.0 * log(u1));
    const double ang = 6.283185307179586476925286766559 * u2;
    r->spare = rad * sin(ang);
    r->have_spare = 1;
    return rad * cos(ang);
}

/* round a double to float, then (optionally) to bf16 with round-to-nearest-even */
static float store_round(double x, int bf16) {
    float f = (float)x;
    if (!bf16) return f;
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u) return f; /* inf / nan unchanged */
    const uint32_t lsb = (u >> 16) & 1u;
    u = (u + 0x7FFFu + lsb) & 0xFFFF0000u;
    memcpy(&f, &u, 4);
    return f;
}

/* kind: 0 = N(mu, sd); 1 = N(0,1) then L2-normalised over groups of `group`;
 *       2 = log(sigmoid(N(mu, sd)));  3 = sigmoid(N(mu, sd))                          */
typedef struct {
    uint64_t seed;
    uint32_t tensor_id;
    long n_rows;
    int row_len, group, kind, bf16;
    double mu, sd;
    float* out;
    long next;
    pthread_mutex_t lock;
} job_t;

static void fill_row(const job_t* j, long row, double* tmp) {
    rng_t r;
    rng_seed(&r, j->seed, j->tensor_id, (uint64_t)row);
    float* o = j->out + (size_t)row * j->row_len;
    for (int i = 0; i < j->row_len; ++i) tmp[i] = rng_normal(&r);
    if (j->kind == 0) {
        for (int i = 0; i < j->row_len; ++i) o[i] = store_round(j->mu + j->sd * tmp[i], j->bf16);
    } else if (j->kind == 1) {
        for (int g0 = 0; g0 < j->row_len; g0 += j->group) {
            double ss = 0.0;
            for (int i = 0; i < j->group; ++i) ss += tmp[g0 + i] * tmp[g0 + i];
            const double inv = 1.0 / sqrt(ss);
            for (int i = 0; i < j->group; ++i) o[g0 + i] = store_round(tmp[g0 + i] * inv, j->bf16);
        }
    } else if (j->kind == 2) {
        for (int i = 0; i < j->row_len; ++i) {
            const double x = j->mu + j->sd * tmp[i];
            /* log(sigmoid(x)) = -log1p(exp(-x)), evaluated without overflow */
            const double ls = (x >= 0.0) ? -log1p(exp(-x)) : x - log1p(exp(x));
            o[i] = store_round(ls, j->bf16);
        }
    } else {
        for (int i = 0; i < j->row_len; ++i) {
            const double x = j->mu + j->sd * tmp[i];
            const double s = (x >= 0.0) ? 1.0 / (1.0 + exp(-x)) : exp(x) / (1.0 + exp(x));
            o[i] = store_round(s, j->bf16);
        }
    }
}

static void* worker(void* arg) {
    job_t* j = (job_t*)arg;
    double* tmp = (double*)malloc(sizeof(double) * (size_t)j->row_len);
    for (;;) {
        pthread_mutex_lock(&j->lock);
        long first = j->next;
        j->next += 64;
        pthread_mutex_unlock(&j->lock);
        if (first >= j->n_rows) break;
        long last = first + 64 < j->n_rows ? first + 64 : j->n_rows;
        for (long r = first; r < last; ++r) fill_row(j, r, tmp);
    }
    free(tmp);
    return NULL;
}

/* Fill out[n_rows * row_len]. Returns 0 on success, -1 on a bad argument. */
int synth_fill(uint64_t seed, uint32_t tensor_id, long n_rows, int row_len, int group, int kind,
               double mu, double sd, int bf16, float* out, int nthreads) {
    if (!out || n_rows < 0 || row_len <= 0 || kind < 0 || kind > 3) return -1;
    if (kind == 1 && (group <= 0 || row_len % group != 0)) return -1;
    job_t j;
    j.seed = seed;
    j.tensor_id = tensor_id;
    j.n_rows = n_rows;
    j.row_len = row_len;
    j.group = group;
    j.kind = kind;
    j.bf16 = bf16;
    j.mu = mu;
    j.sd = sd;
    j.out = out;
    j.next = 0;
    pthread_mutex_init(&j.lock, NULL);
    int nt = nthreads;
    if (nt <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nt = n > 0 ? (int)n : 1;
    }
    long max_nt = (n_rows + 63) / 64;
    if (nt > max_nt) nt = (int)(max_nt > 0 ? max_nt : 1);
    if (nt <= 1) {
        worker(&j);
    } else {
        pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nt);
        for (int i = 0; i < nt; ++i) pthread_create(&th[i], NULL, worker, &j);
        for (int i = 0; i < nt; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&j.lock);
    return 0;
}
