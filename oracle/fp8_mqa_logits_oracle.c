/*
 * CPU oracle for the prefill FP8 MQA indexer logits -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the bench's CPU-baseline leg may load this
 * file's library.  The product path (the CUDA library) never calls it, and the two
 * share no code, header, table or constant.
 *
 * What it computes (ROCm/aiter PR #7183 "[HIP] [JIT] Add gfx950 prefill FP8 MQA
 * logits", section "Motivation", the displayed formula):
 *
 *     logits[m, n] = sum_h relu( Q[m,h,:] . K[n,:] ) * w[m,h] * kv_scale[n]
 *                    for n in [ks[m], ke[m]),   -inf elsewhere
 *
 * The operator contract (same page, "PR-specific question"): FP8 Q/K, float32
 * scales and weights, int32 row bounds, contiguous row-major layouts.  The page
 * calls the inputs "FP8" only; this oracle reads that as OCP E4M3 ("e4m3fn":
 * 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, subnormals at exponent
 * 0, S.1111.111 = NaN, no infinities, largest finite value 448).
 *
 * Every step is the plain definition, in fp64, in the page's order: decode, dot
 * over d, relu, times w, sum over h, times kv_scale.  Readings taken where the
 * page is silent:
 *   - the window is half-open and clamped to [0, N); ks >= ke is an empty row;
 *   - clean_logits = 1 writes -inf outside the window; clean_logits = 0 leaves
 *     those entries of `out` exactly as the caller left them ("caller-managed
 *     output masks", page section "PR Self-Review / Behavior and intent");
 *   - kv_scale multiplies after the head sum, as the formula is written.
 *
 * Exactness note: every finite e4m3 value is an integer multiple of 2^-9 with
 * magnitude <= 448, so each product is a multiple of 2^-18 and any dot over
 * D <= 2^12 terms stays below 2^53 * 2^-18: the fp64 dot is exact.  Only the
 * products by w and kv_scale and the head sum round, at about 1e-16 relative.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Decode one OCP E4M3 byte to double, from the bit-field definition. */
static double e4m3_decode(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int exp = (b >> 3) & 0xF;
    int man = b & 0x7;
    double v;
    if (exp == 0xF && man == 0x7) {
        v = NAN; /* S.1111.111 is the only NaN pattern; there is no infinity */
    } else if (exp == 0) {
        v = ldexp((double)man / 8.0, 1 - 7); /* subnormal: 0.mmm * 2^(1-bias) */
    } else {
        v = ldexp(1.0 + (double)man / 8.0, exp - 7); /* normal: 1.mmm * 2^(e-bias) */
    }
    return sign ? -v : v;
}

void oracle_e4m3_table(double table[256])
{
    for (int i = 0; i < 256; ++i) table[i] = e4m3_decode((uint8_t)i);
}

typedef struct {
    const uint8_t* q;
    const uint8_t* k;
    const float* kv_scale;
    const float* w;
    const int32_t* ks;
    const int32_t* ke;
    double* out;
    const int64_t* rows; /* NULL: all rows 0..M-1, out is [M, N]; else out is [nrows, N] */
    int64_t nrows;
    int64_t M, N;
    int32_t H, D;
    int32_t clean;
    int32_t tid, nthreads;
    double table[256];
} oracle_job;

/* One output row: the formula above for query row m, written into out_row[0..N). */
static void oracle_row(const oracle_job* j, int64_t m, double* out_row)
{
    const int64_t N = j->N;
    const int32_t H = j->H, D = j->D;
    int64_t lo = j->ks[m], hi = j->ke[m];
    if (lo < 0) lo = 0;
    if (hi > N) hi = N;
    for (int64_t n = 0; n < N; ++n) {
        if (n < lo || n >= hi) {
            if (j->clean) out_row[n] = -INFINITY; /* outside the window */
            continue;                             /* clean = 0: untouched */
        }
        double acc = 0.0;
        for (int32_t h = 0; h < H; ++h) {
            const uint8_t* qv = j->q + ((size_t)m * H + h) * D;
            const uint8_t* kv = j->k + (size_t)n * D;
            double dot = 0.0;
            for (int32_t d = 0; d < D; ++d) dot += j->table[qv[d]] * j->table[kv[d]];
            double r = dot > 0.0 ? dot : 0.0; /* relu */
            acc += r * (double)j->w[(size_t)m * H + h];
        }
        out_row[n] = acc * (double)j->kv_scale[n];
    }
}

static void* oracle_worker(void* arg)
{
    const oracle_job* j = (const oracle_job*)arg;
    const int64_t count = j->rows ? j->nrows : j->M;
    for (int64_t i = j->tid; i < count; i += j->nthreads) {
        int64_t m = j->rows ? j->rows[i] : i;
        oracle_row(j, m, j->out + (size_t)i * j->N);
    }
    return NULL;
}

/*
 * Host pointers throughout.  q: [M,H,D] bytes, k: [N,D] bytes, kv_scale: [N],
 * w: [M,H], ks/ke: [M], out: [M,N] fp64 (or [nrows,N] when rows != NULL, holding
 * the rows listed in `rows`).  Returns 0, or -1 on a bad argument.
 */
int oracle_fp8_mqa_logits(const uint8_t* q, const uint8_t* k, const float* kv_scale,
                          const float* w, const int32_t* ks, const int32_t* ke, double* out,
                          int64_t M, int64_t N, int32_t H, int32_t D, int32_t clean_logits,
                          const int64_t* rows, int64_t nrows, int32_t nthreads)
{
    if (M < 0 || N < 0 || H <= 0 || D <= 0 || nrows < 0) return -1;
    if (rows) {
        for (int64_t i = 0; i < nrows; ++i)
            if (rows[i] < 0 || rows[i] >= M) return -1;
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;

    oracle_job* jobs = (oracle_job*)malloc(sizeof(oracle_job) * (size_t)nthreads);
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -1;
    }
    for (int32_t t = 0; t < nthreads; ++t) {
        oracle_job* j = &jobs[t];
        j->q = q; j->k = k; j->kv_scale = kv_scale; j->w = w; j->ks = ks; j->ke = ke;
        j->out = out; j->rows = rows; j->nrows = nrows; j->M = M; j->N = N;
        j->H = H; j->D = D; j->clean = clean_logits ? 1 : 0;
        j->tid = t; j->nthreads = nthreads;
        oracle_e4m3_table(j->table);
    }
    int32_t started = 0;
    for (int32_t t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, oracle_worker, &jobs[t]) != 0) break;
        started = t;
    }
    /* threads that failed to start: fold their rows into the calling thread */
    if (started < nthreads - 1) {
        for (int32_t t = started + 1; t < nthreads; ++t) oracle_worker(&jobs[t]);
    }
    oracle_worker(&jobs[0]);
    for (int32_t t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    free(jobs);
    free(th);
    return 0;
}
