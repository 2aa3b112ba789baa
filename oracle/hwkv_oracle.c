/*
 * Oracle for per-head windowed decode attention -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow fp64 restatement of what HeadWiseKV's grouped-cache runtime computes
 * for one decode step (HeadWiseKV blog summary, abstract: each physical KV head keeps a
 * static window of its most recent tokens, and the runtime materialises that residency
 * instead of masking a full cache; section "Grouped-Cache Runtime").  Because
 * materialising and masking reach the same result, the oracle is the masked definition
 * written out over the FULL token history -- it never looks at a pool, a block table or
 * a ring slot:
 *
 *     P   = [max(0, len - w), len)                  (the last min(w, len) positions)
 *     s_p = scale * sum_d q[d] * k[p][d]
 *     o   = sum_p exp(s_p - max s) v[p] / sum_p exp(s_p - max s)
 *
 * An empty window (len == 0) yields a zero vector.  bf16 inputs are widened exactly to
 * fp64.  Shares no code with the CUDA library; only tests/, the smoke check and the
 * benchmark's CPU baseline load it.
 */
#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F64 = 2 };

typedef struct {
    const void* q;       /* [head_dim] query vector of one query head                 */
    const void* k;       /* history rows, row i = position p_lo + i, row_stride elems */
    const void* v;
    int64_t row_stride;  /* elements between consecutive history rows                 */
    int64_t p_lo;        /* first position present in k / v                           */
    int64_t n_hist;      /* number of history rows present                            */
    int64_t len;         /* sequence length (positions 0 .. len-1 exist)              */
    int64_t window;      /* static window w of the KV head                            */
    double scale;
    double* out;         /* [head_dim] fp64 result                                    */
} oracle_attn_job;

static double widen(const void* base, int64_t i, int dtype) {
    if (dtype == ORACLE_F32) return (double)((const float*)base)[i];
    if (dtype == ORACLE_F64) return ((const double*)base)[i];
    uint32_t bits = (uint32_t)((const uint16_t*)base)[i] << 16; /* bf16 -> fp32 bits */
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* returns 0, or -1 when the window is not covered by the history passed in */
static int attend_one(const oracle_attn_job* j, int D, int dtype, double* scores) {
    int64_t lo = j->len - j->window;
    if (lo < 0) lo = 0;
    int64_t hi = j->len;
    for (int d = 0; d < D; ++d) j->out[d] = 0.0;
    if (hi <= lo) return 0;
    if (lo < j->p_lo || hi > j->p_lo + j->n_hist) return -1;

    double m = -INFINITY;
    for (int64_t p = lo; p < hi; ++p) {
        int64_t row = (p - j->p_lo) * j->row_stride;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += widen(j->q, d, dtype) * widen(j->k, row + d, dtype);
        double s = j->scale * dot;
        scores[p - lo] = s;
        if (s > m) m = s;
    }
    double z = 0.0;
    for (int64_t p = lo; p < hi; ++p) {
        int64_t row = (p - j->p_lo) * j->row_stride;
        double e = exp(scores[p - lo] - m);
        z += e;
        for (int d = 0; d < D; ++d) j->out[d] += e * widen(j->v, row + d, dtype);
    }
    for (int d = 0; d < D; ++d) j->out[d] /= z;
    return 0;
}

typedef struct {
    const oracle_attn_job* jobs;
    int64_t n_jobs;
    int D, dtype;
    int64_t max_window;
    atomic_long next;
    atomic_int status;
} shared_t;

static void* worker(void* arg) {
    shared_t* sh = (shared_t*)arg;
    double* scores = (double*)malloc(sizeof(double) * (size_t)(sh->max_window > 0 ? sh->max_window : 1));
    if (!scores) { atomic_store(&sh->status, -2); return NULL; }
    for (;;) {
        long i = atomic_fetch_add(&sh->next, 1);
        if (i >= sh->n_jobs) break;
        if (attend_one(&sh->jobs[i], sh->D, sh->dtype, scores) != 0) atomic_store(&sh->status, -1);
    }
    free(scores);
    return NULL;
}

/* Runs every job; threads <= 0 means one.  Returns 0, -1 (history does not cover a
 * window), -2 (out of memory) or -3 (bad arguments). */
int oracle_attention(const oracle_attn_job* jobs, int64_t n_jobs, int head_dim, int dtype, int threads) {
    if (n_jobs < 0 || head_dim <= 0 || (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F64))
        return -3;
    shared_t sh;
    sh.jobs = jobs;
    sh.n_jobs = n_jobs;
    sh.D = head_dim;
    sh.dtype = dtype;
    sh.max_window = 1;
    for (int64_t i = 0; i < n_jobs; ++i) {
        int64_t n = jobs[i].window < jobs[i].len ? jobs[i].window : jobs[i].len;
        if (n > sh.max_window) sh.max_window = n;
    }
    atomic_init(&sh.next, 0);
    atomic_init(&sh.status, 0);
    if (threads <= 1) {
        worker(&sh);
        return atomic_load(&sh.status);
    }
    pthread_t* tid = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)threads);
    if (!tid) return -2;
    int started = 0;
    for (int t = 0; t < threads; ++t)
        if (pthread_create(&tid[t], NULL, worker, &sh) == 0) ++started;
    if (started == 0) worker(&sh);
    for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    free(tid);
    return atomic_load(&sh.status);
}

int oracle_abi(void) { return 1; }
